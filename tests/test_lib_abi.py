"""libhb.so loads, exports every entry point include/hb.h declares, and its
host-side validation rejects bad arguments before touching CUDA (CPU only:
no call here reaches a kernel launch or any CUDA runtime call)."""

import ctypes
import os
import re
import subprocess

import pytest

from linear_attention_diffusion_feature_b300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hb.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hb_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("hb_feature_map", "hb_block_attend", "hb_commit_block", "hb_prefill_state",
                     "hb_softmax_kv_attend", "hb_state_zero", "hb_get_device_status"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (hb_[a-z0-9_]+)\b", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for name in declared_functions():
        assert hasattr(lib, name)


def test_binding_covers_exactly_the_header():
    assert sorted(_lib.SIGNATURES) == declared_functions()


def test_library_has_no_driver_or_torch_dependency():
    out = subprocess.run(["ldd", _lib.LIB_PATH], capture_output=True, text=True).stdout
    assert "libtorch" not in out and "libc10" not in out


def test_status_strings(lib):
    for code in range(8):
        s = lib.hb_status_string(code)
        assert s and s != b"unknown status"
    assert lib.hb_status_string(99) == b"unknown status"


def _cfg(**kw):
    base = dict(num_heads=16, head_dim=128, feat_half=64, block_len=32, dtype=0, merge=0, scale=0.0)
    base.update(kw)
    return _lib.HBConfig(**base)


# Fake, never dereferenced device addresses: validation fails or returns
# early before any pointer is used.
A = ctypes.c_void_p(0x10000)      # 16-byte aligned
M = ctypes.c_void_p(0x10008)      # misaligned


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=8), 2), (dict(head_dim=136), 2), (dict(head_dim=72), 2),
    (dict(feat_half=4), 2), (dict(feat_half=72), 2), (dict(feat_half=12), 2),
    (dict(block_len=0), 2), (dict(block_len=65), 2), (dict(num_heads=0), 2),
    (dict(dtype=7), 1), (dict(merge=3), 1), (dict(scale=-1.0), 1),
    (dict(scale=float("inf")), 1), (dict(scale=float("nan")), 1),
])
def test_attend_rejects_bad_config(lib, kw, code):
    c = _cfg(**kw)
    r = lib.hb_block_attend(ctypes.byref(c), 1, A, A, A, A, A, A, 1, A, A, A, None)
    assert r == code


def test_attend_null_config(lib):
    assert lib.hb_block_attend(None, 1, A, A, A, A, A, A, 1, A, A, A, None) == 1


def test_attend_pointer_checks(lib):
    c = _cfg()
    assert lib.hb_block_attend(ctypes.byref(c), 1, A, None, A, A, A, A, 1, A, A, A, None) == 1
    assert lib.hb_block_attend(ctypes.byref(c), 1, A, A, A, M, A, A, 1, A, A, A, None) == 3
    assert lib.hb_block_attend(ctypes.byref(c), -1, A, A, A, A, A, A, 1, A, A, A, None) == 1
    # batch 0 is a no-op that succeeds without looking at the pointers
    assert lib.hb_block_attend(ctypes.byref(c), 0, None, None, None, None, None, None, 0, None,
                               None, None, None) == 0


def test_attend_layers_checks(lib):
    c = _cfg()
    f = lib.hb_block_attend_commit_layers
    # n_layers must be >= 1
    assert f(ctypes.byref(c), 0, 2, A, A, A, A, A, A, 4, A, A, A, A, None) == 1
    assert f(ctypes.byref(c), -3, 2, A, A, A, A, A, A, 4, A, A, A, A, None) == 1
    # a null or misaligned operand; the commit mask may be null (attend only)
    assert f(ctypes.byref(c), 6, 2, A, A, None, A, A, A, 4, A, A, A, A, None) == 1
    assert f(ctypes.byref(c), 6, 2, A, A, A, A, M, A, 4, A, A, A, A, None) == 3
    assert f(ctypes.byref(c), 6, -1, A, A, A, A, A, A, 4, A, A, A, A, None) == 1
    # more requests in one call than the kernels index
    assert f(ctypes.byref(c), 64, 65535, A, A, A, A, A, A, 4, A, A, A, A, None) == 2
    # batch 0 is a no-op
    assert f(ctypes.byref(c), 6, 0, None, None, None, None, None, None, 0, None, None, None,
             None, None) == 0


def test_attend_layers_binding_rejects_a_ragged_split():
    import torch

    import linear_attention_diffusion_feature_b300 as hb
    cfg = hb.Config(16, 128, 64, 32)
    W = torch.zeros((3, 16, 128, 64), dtype=torch.bfloat16)
    sl = torch.zeros((8,), dtype=torch.int32)  # 8 requests do not split into 3 layers
    with pytest.raises(ValueError):
        hb.hb_block_attend_commit_layers(cfg, sl, None, None, None, None, None, W, None)


def test_commit_and_zero_checks(lib):
    c = _cfg()
    assert lib.hb_commit_block(ctypes.byref(c), 2, A, A, None, A, A, A, 4, None) == 1
    assert lib.hb_commit_block(ctypes.byref(c), 2, A, A, A, A, M, A, 4, None) == 3
    assert lib.hb_commit_block(ctypes.byref(c), 0, None, None, None, None, None, None, 0, None) == 0
    assert lib.hb_state_zero(ctypes.byref(c), 1, A, None, A, 1, None) == 1
    assert lib.hb_state_zero(ctypes.byref(c), 0, None, None, None, 0, None) == 0


def test_prefill_checks(lib):
    c = _cfg()
    # negative sizes, bad accumulate flag
    assert lib.hb_prefill_state(ctypes.byref(c), 1, A, A, A, -1, A, 8, A, A, A, 1, 0, None, 0,
                                None) == 1
    assert lib.hb_prefill_state(ctypes.byref(c), 1, A, A, A, 8, A, -8, A, A, A, 1, 0, None, 0,
                                None) == 1
    assert lib.hb_prefill_state(ctypes.byref(c), 1, A, A, A, 8, A, 8, A, A, A, 1, 2, None, 0,
                                None) == 1
    # tokens present but k missing
    assert lib.hb_prefill_state(ctypes.byref(c), 1, A, None, A, 8, A, 8, A, A, A, 1, 0, None, 0,
                                None) == 1
    need = lib.hb_prefill_workspace_size(ctypes.byref(c), 8, 8192)
    if need:
        assert lib.hb_prefill_state(ctypes.byref(c), 8, A, A, A, 65536, A, 8192, A, A, A, 8, 0,
                                    A, need - 16, None) == 7


def test_prefill_attend_checks(lib):
    c = _cfg()
    # args: cfg, batch, slot_idx, q, k, v, seq_len, S, Z, num_slots, W, gate, accumulate, o, stream
    # prompt length not a multiple of the block length (32)
    assert lib.hb_prefill_attend(ctypes.byref(c), 1, A, A, A, A, 33, A, A, 1, A, A, 0, A,
                                 None) == 1
    assert lib.hb_prefill_attend(ctypes.byref(c), 1, A, A, A, A, -32, A, A, 1, A, A, 0, A,
                                 None) == 1
    # bad accumulate flag, missing q, misaligned o
    assert lib.hb_prefill_attend(ctypes.byref(c), 1, A, A, A, A, 64, A, A, 1, A, A, 2, A,
                                 None) == 1
    assert lib.hb_prefill_attend(ctypes.byref(c), 1, A, None, A, A, 64, A, A, 1, A, A, 0, A,
                                 None) == 1
    assert lib.hb_prefill_attend(ctypes.byref(c), 1, A, A, A, A, 64, A, A, 1, A, A, 0, M,
                                 None) == 3
    # batch 0 is a no-op
    assert lib.hb_prefill_attend(ctypes.byref(c), 0, None, None, None, None, 64, None, None, 0,
                                 None, None, 0, None, None) == 0


def test_softmax_kv_checks(lib):
    c = _cfg()
    assert lib.hb_softmax_kv_attend(ctypes.byref(c), 1, A, A, 8, None, 8, A, A, A, A, None, 0,
                                    None) == 1
    assert lib.hb_softmax_kv_attend(ctypes.byref(c), 1, None, A, 8, A, 8, A, A, A, A, None, 0,
                                    None) == 1
    assert lib.hb_softmax_kv_attend(ctypes.byref(c), 1, A, A, 8, A, 8, A, M, A, A, None, 0,
                                    None) == 3


def test_softmax_kv_paged_checks(lib):
    c = _cfg()
    # args: cfg, batch, k_pages, v_pages, num_pages, page_tokens, page_table, max_pages,
    #       prefix_len, max_prefix, q, k, v, o, workspace, workspace_bytes, stream
    def call(batch=1, num_pages=4, page_tokens=32, table=A, max_pages=2, plen=A,
             max_prefix=64, q=A, kp=A):
        return lib.hb_softmax_kv_attend_paged(ctypes.byref(c), batch, kp, kp, num_pages,
                                              page_tokens, table, max_pages, plen, max_prefix,
                                              q, A, A, A, None, 0, None)
    assert call(batch=-1) == 1
    assert call(page_tokens=0) == 1
    assert call(num_pages=-1) == 1
    assert call(max_pages=-1) == 1
    assert call(max_prefix=-1) == 1
    assert call(max_prefix=1 << 31) == 1          # prefix lengths are int32
    assert call(plen=None) == 1
    assert call(table=None) == 1                  # pages to look up but no table
    assert call(kp=None) == 1                     # a non-empty pool needs its pointers
    assert call(q=M) == 3
    assert call(table=M) == 3
    assert call(batch=0, table=None, plen=None, q=None, kp=None) == 0


def test_state_copy_checks(lib):
    c = _cfg()
    # args: cfg, batch, src_slot, dst_slot, S, Z, num_slots, stream
    assert lib.hb_state_copy(ctypes.byref(c), -1, A, A, A, A, 4, None) == 1
    assert lib.hb_state_copy(ctypes.byref(c), 1, A, A, A, A, -1, None) == 1
    assert lib.hb_state_copy(ctypes.byref(c), 1, None, A, A, A, 4, None) == 1
    assert lib.hb_state_copy(ctypes.byref(c), 1, A, A, M, A, 4, None) == 3
    assert lib.hb_state_copy(ctypes.byref(_cfg(head_dim=8)), 1, A, A, A, A, 4, None) == 2
    assert lib.hb_state_copy(ctypes.byref(c), 0, None, None, None, None, 0, None) == 0


def test_state_bf16_copy_checks(lib):
    c = _cfg()
    # hb_state_to_bf16: cfg, batch, slot_idx, S, S16, num_slots, stream
    assert lib.hb_state_to_bf16(ctypes.byref(c), -1, A, A, A, 4, None) == 1
    assert lib.hb_state_to_bf16(ctypes.byref(c), 1, A, A, None, 4, None) == 1
    assert lib.hb_state_to_bf16(ctypes.byref(c), 1, A, M, A, 4, None) == 3
    assert lib.hb_state_to_bf16(ctypes.byref(c), 0, None, None, None, 0, None) == 0
    # hb_block_attend_s16: cfg, batch, slot_idx, q, k, v, S16, Z, num_slots, W, gate, o, stream
    args = (A, A, A, A, A, A, 4, A, A, A, None)
    assert lib.hb_block_attend_s16(ctypes.byref(c), -1, *args) == 1
    assert lib.hb_block_attend_s16(ctypes.byref(_cfg(head_dim=64)), 1, *args) == 2
    assert lib.hb_block_attend_s16(ctypes.byref(_cfg(dtype=1)), 1, *args) == 2
    assert lib.hb_block_attend_s16(ctypes.byref(c), 1, A, A, A, A, None, A, 4, A, A, A,
                                   None) == 1
    assert lib.hb_block_attend_s16(ctypes.byref(c), 1, A, A, A, A, M, A, 4, A, A, A,
                                   None) == 3
    assert lib.hb_block_attend_s16(ctypes.byref(c), 0, *args) == 0


def test_feature_map_checks(lib):
    c = _cfg()
    assert lib.hb_feature_map(ctypes.byref(c), -1, A, A, A, None) == 1
    assert lib.hb_feature_map(ctypes.byref(c), 0, None, A, None, None) == 0
    assert lib.hb_feature_map(ctypes.byref(c), 4, A, M, A, None) == 3
    assert lib.hb_feature_map(ctypes.byref(_cfg(feat_half=100)), 4, A, A, A, None) == 2


def test_workspace_size_queries_reject_bad_args(lib):
    assert lib.hb_prefill_workspace_size(None, 8, 8192) == 0
    assert lib.hb_prefill_workspace_size(ctypes.byref(_cfg(head_dim=8)), 8, 8192) == 0
    assert lib.hb_softmax_kv_workspace_size(ctypes.byref(_cfg()), -1, 2048) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "libhb.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        _lib.load()
