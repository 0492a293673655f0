"""Python binding of libhb.so with the C ABI's names (include/hb.h).

Argument marshalling only: every function checks that the torch tensors it is
given live on the current CUDA device with the dtype, shape and contiguity the
C ABI expects (a wrong size would otherwise become an out-of-bounds access on
the device), passes their pointers and the current stream to the library, and
raises ``HBError`` on a non-zero status. All arithmetic runs in the CUDA
kernels of libhb.so; there is no other implementation to fall back to.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib

DTYPE_BF16 = 0
DTYPE_FP32 = 1
MERGE_SHARED_NORM = 0
MERGE_CONVEX = 1

_TORCH_DTYPE = {DTYPE_BF16: torch.bfloat16, DTYPE_FP32: torch.float32}


class HBError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _lib.load()
        msg = lib.hb_status_string(status).decode()
        super().__init__(f"{where}: {_lib.STATUS_NAMES.get(status, status)} ({msg})")
        self.status = status


@dataclass(frozen=True)
class Config:
    """``hb_config``: H heads, head dim d, half feature width f (F = 2f),
    block length L, activation dtype, merge form, block softmax scale
    (0 means 1/sqrt(d))."""

    num_heads: int
    head_dim: int
    feat_half: int
    block_len: int
    dtype: int = DTYPE_BF16
    merge: int = MERGE_SHARED_NORM
    scale: float = 0.0

    @property
    def F(self) -> int:
        return 2 * self.feat_half

    @property
    def torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPE[self.dtype]

    def c(self) -> _lib.HBConfig:
        return _lib.HBConfig(self.num_heads, self.head_dim, self.feat_half, self.block_len,
                             self.dtype, self.merge, self.scale)


def _check(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor, got {t.device}")
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        # the library launches on the current device; a pointer into another
        # GPU's memory would be dereferenced there
        raise ValueError(f"{name}: lives on {t.device}, but the current device is cuda:{cur}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    cur = torch.cuda.current_device()
    if s.device.index != cur:
        raise ValueError(f"stream belongs to {s.device}, but the current device is cuda:{cur}")
    return ctypes.c_void_p(s.cuda_stream)


def _raise(status: int, where: str) -> None:
    if status != _lib.HB_OK:
        raise HBError(status, where)


def hb_feature_map(cfg: Config, x: torch.Tensor, W: torch.Tensor, phi: torch.Tensor = None,
                   stream=None) -> torch.Tensor:
    """phi(x) = [softmax(x W_h), softmax(-x W_h)]: x [n, H, d] -> phi [n, H, 2f] fp32."""
    n = x.shape[0]
    H, d, f = cfg.num_heads, cfg.head_dim, cfg.feat_half
    _check(x, "x", cfg.torch_dtype, (n, H, d))
    _check(W, "W", cfg.torch_dtype, (H, d, f))
    if phi is None:
        phi = torch.empty((n, H, 2 * f), dtype=torch.float32, device=x.device)
    _check(phi, "phi", torch.float32, (n, H, 2 * f))
    lib = _lib.load()
    _raise(lib.hb_feature_map(ctypes.byref(cfg.c()), n, _ptr(x), _ptr(W), _ptr(phi),
                              _stream(stream)), "hb_feature_map")
    return phi


def _check_state(cfg, S_pool, Z_pool):
    if S_pool.dim() != 4:
        raise ValueError("S_pool: expected [num_slots, H, F, d]")
    num_slots = S_pool.shape[0]
    _check(S_pool, "S_pool", torch.float32, (num_slots, cfg.num_heads, cfg.F, cfg.head_dim))
    _check(Z_pool, "Z_pool", torch.float32, (num_slots, cfg.num_heads, cfg.F))
    return num_slots


def hb_block_attend(cfg: Config, slot_idx, q, k, v, S_pool, Z_pool, W, gate_logits, o=None,
                    stream=None) -> torch.Tensor:
    """Block-hybrid attention of the active block: q/k/v [B, L, H, d] -> o."""
    B = slot_idx.shape[0]
    H, d, f, L = cfg.num_heads, cfg.head_dim, cfg.feat_half, cfg.block_len
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, cfg.torch_dtype, (B, L, H, d))
    num_slots = _check_state(cfg, S_pool, Z_pool)
    _check(W, "W", cfg.torch_dtype, (H, d, f))
    _check(gate_logits, "gate_logits", torch.float32, (H,))
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", cfg.torch_dtype, (B, L, H, d))
    lib = _lib.load()
    _raise(lib.hb_block_attend(ctypes.byref(cfg.c()), B, _ptr(slot_idx), _ptr(q), _ptr(k),
                               _ptr(v), _ptr(S_pool), _ptr(Z_pool), num_slots, _ptr(W),
                               _ptr(gate_logits), _ptr(o), _stream(stream)), "hb_block_attend")
    return o


def hb_state_to_bf16(cfg: Config, slot_idx, S_pool, S16_pool, stream=None) -> None:
    """Writes the bf16 copy of the listed slots' S (round to nearest) that
    hb_block_attend_s16 reads."""
    B = slot_idx.shape[0]
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    if S_pool.dim() != 4:
        raise ValueError("S_pool: expected [num_slots, H, F, d]")
    num_slots = S_pool.shape[0]
    shape = (num_slots, cfg.num_heads, cfg.F, cfg.head_dim)
    _check(S_pool, "S_pool", torch.float32, shape)
    _check(S16_pool, "S16_pool", torch.bfloat16, shape)
    lib = _lib.load()
    _raise(lib.hb_state_to_bf16(ctypes.byref(cfg.c()), B, _ptr(slot_idx), _ptr(S_pool),
                                _ptr(S16_pool), num_slots, _stream(stream)), "hb_state_to_bf16")


def hb_block_attend_s16(cfg: Config, slot_idx, q, k, v, S16_pool, Z_pool, W, gate_logits,
                        o=None, stream=None) -> torch.Tensor:
    """hb_block_attend on the bf16 copy of S (bit-identical output, half the
    state bytes); Z_pool is the fp32 master's."""
    B = slot_idx.shape[0]
    H, d, f, L = cfg.num_heads, cfg.head_dim, cfg.feat_half, cfg.block_len
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, cfg.torch_dtype, (B, L, H, d))
    if S16_pool.dim() != 4:
        raise ValueError("S16_pool: expected [num_slots, H, F, d]")
    num_slots = S16_pool.shape[0]
    _check(S16_pool, "S16_pool", torch.bfloat16, (num_slots, H, cfg.F, d))
    _check(Z_pool, "Z_pool", torch.float32, (num_slots, H, cfg.F))
    _check(W, "W", cfg.torch_dtype, (H, d, f))
    _check(gate_logits, "gate_logits", torch.float32, (H,))
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", cfg.torch_dtype, (B, L, H, d))
    lib = _lib.load()
    _raise(lib.hb_block_attend_s16(ctypes.byref(cfg.c()), B, _ptr(slot_idx), _ptr(q), _ptr(k),
                                   _ptr(v), _ptr(S16_pool), _ptr(Z_pool), num_slots, _ptr(W),
                                   _ptr(gate_logits), _ptr(o), _stream(stream)),
           "hb_block_attend_s16")
    return o


def hb_state_to_fp8(cfg: Config, slot_idx, S_pool, S8_pool, scale_pool, stream=None) -> None:
    """Writes the fp8 (e4m3) copy of the listed slots' S, one scale per
    (slot, head): scale = max|S| / 448, code = e4m3(S / scale)."""
    B = slot_idx.shape[0]
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    if S_pool.dim() != 4:
        raise ValueError("S_pool: expected [num_slots, H, F, d]")
    num_slots = S_pool.shape[0]
    shape = (num_slots, cfg.num_heads, cfg.F, cfg.head_dim)
    _check(S_pool, "S_pool", torch.float32, shape)
    _check(S8_pool, "S8_pool", torch.uint8, shape)
    _check(scale_pool, "scale_pool", torch.float32, (num_slots, cfg.num_heads))
    lib = _lib.load()
    _raise(lib.hb_state_to_fp8(ctypes.byref(cfg.c()), B, _ptr(slot_idx), _ptr(S_pool),
                               _ptr(S8_pool), _ptr(scale_pool), num_slots, _stream(stream)),
           "hb_state_to_fp8")


def hb_block_attend_s8(cfg: Config, slot_idx, q, k, v, S8_pool, scale_pool, Z_pool, W,
                       gate_logits, o=None, stream=None) -> torch.Tensor:
    """hb_block_attend on the fp8 copy of S (a quarter of the state bytes;
    the output is the attend on the dequantised state); Z_pool is the fp32
    master's."""
    B = slot_idx.shape[0]
    H, d, f, L = cfg.num_heads, cfg.head_dim, cfg.feat_half, cfg.block_len
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, cfg.torch_dtype, (B, L, H, d))
    if S8_pool.dim() != 4:
        raise ValueError("S8_pool: expected [num_slots, H, F, d]")
    num_slots = S8_pool.shape[0]
    _check(S8_pool, "S8_pool", torch.uint8, (num_slots, H, cfg.F, d))
    _check(scale_pool, "scale_pool", torch.float32, (num_slots, H))
    _check(Z_pool, "Z_pool", torch.float32, (num_slots, H, cfg.F))
    _check(W, "W", cfg.torch_dtype, (H, d, f))
    _check(gate_logits, "gate_logits", torch.float32, (H,))
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", cfg.torch_dtype, (B, L, H, d))
    lib = _lib.load()
    _raise(lib.hb_block_attend_s8(ctypes.byref(cfg.c()), B, _ptr(slot_idx), _ptr(q), _ptr(k),
                                  _ptr(v), _ptr(S8_pool), _ptr(scale_pool), _ptr(Z_pool),
                                  num_slots, _ptr(W), _ptr(gate_logits), _ptr(o),
                                  _stream(stream)), "hb_block_attend_s8")
    return o


def hb_block_attend_commit(cfg: Config, slot_idx, q, k, v, S_pool, Z_pool, W, gate_logits,
                           commit, o=None, stream=None) -> torch.Tensor:
    """hb_block_attend, then hb_commit_block of the same block for the requests
    with commit[b] != 0, in one pass over the state."""
    B = slot_idx.shape[0]
    H, d, f, L = cfg.num_heads, cfg.head_dim, cfg.feat_half, cfg.block_len
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    _check(commit, "commit", torch.int32, (B,))
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, cfg.torch_dtype, (B, L, H, d))
    num_slots = _check_state(cfg, S_pool, Z_pool)
    _check(W, "W", cfg.torch_dtype, (H, d, f))
    _check(gate_logits, "gate_logits", torch.float32, (H,))
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", cfg.torch_dtype, (B, L, H, d))
    lib = _lib.load()
    _raise(lib.hb_block_attend_commit(ctypes.byref(cfg.c()), B, _ptr(slot_idx), _ptr(q), _ptr(k),
                                      _ptr(v), _ptr(S_pool), _ptr(Z_pool), num_slots, _ptr(W),
                                      _ptr(gate_logits), _ptr(commit), _ptr(o), _stream(stream)),
           "hb_block_attend_commit")
    return o


def hb_block_attend_commit_layers(cfg: Config, slot_idx, q, k, v, S_pool, Z_pool, W,
                                  gate_logits, commit=None, o=None, stream=None) -> torch.Tensor:
    """The fused step of several independent layers in one call: W is
    [n_layers, H, d, f], gate_logits [n_layers, H]; q, k, v, o, slot_idx and
    commit (None: attend only) hold n_layers x batch requests, layer by
    layer."""
    Lyr = W.shape[0] if W.dim() == 4 else 0
    R = slot_idx.shape[0]
    H, d, f, L = cfg.num_heads, cfg.head_dim, cfg.feat_half, cfg.block_len
    if Lyr < 1 or R % Lyr != 0:
        raise ValueError("W must be [n_layers, H, d, f] with n_layers dividing the requests")
    B = R // Lyr
    _check(slot_idx, "slot_idx", torch.int32, (R,))
    if commit is not None:
        _check(commit, "commit", torch.int32, (R,))
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, cfg.torch_dtype, (R, L, H, d))
    num_slots = _check_state(cfg, S_pool, Z_pool)
    _check(W, "W", cfg.torch_dtype, (Lyr, H, d, f))
    _check(gate_logits, "gate_logits", torch.float32, (Lyr, H))
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", cfg.torch_dtype, (R, L, H, d))
    lib = _lib.load()
    _raise(lib.hb_block_attend_commit_layers(
        ctypes.byref(cfg.c()), Lyr, B, _ptr(slot_idx), _ptr(q), _ptr(k), _ptr(v), _ptr(S_pool),
        _ptr(Z_pool), num_slots, _ptr(W), _ptr(gate_logits),
        _ptr(commit), _ptr(o), _stream(stream)),
        "hb_block_attend_commit_layers")
    return o


def hb_block_attend_commit_s16(cfg: Config, slot_idx, q, k, v, S_pool, S16_pool, Z_pool, W,
                               gate_logits, commit, o=None, stream=None) -> torch.Tensor:
    """hb_block_attend_commit on a pool with bf16 copies beside the fp32
    masters: requests that do not commit read their copy, committing ones
    read the master and write the new master and copy."""
    B = slot_idx.shape[0]
    H, d, f, L = cfg.num_heads, cfg.head_dim, cfg.feat_half, cfg.block_len
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    _check(commit, "commit", torch.int32, (B,))
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, cfg.torch_dtype, (B, L, H, d))
    num_slots = _check_state(cfg, S_pool, Z_pool)
    _check(S16_pool, "S16_pool", torch.bfloat16, (num_slots, H, cfg.F, d))
    _check(W, "W", cfg.torch_dtype, (H, d, f))
    _check(gate_logits, "gate_logits", torch.float32, (H,))
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", cfg.torch_dtype, (B, L, H, d))
    lib = _lib.load()
    _raise(lib.hb_block_attend_commit_s16(ctypes.byref(cfg.c()), B, _ptr(slot_idx), _ptr(q),
                                          _ptr(k), _ptr(v), _ptr(S_pool), _ptr(S16_pool),
                                          _ptr(Z_pool), num_slots, _ptr(W), _ptr(gate_logits),
                                          _ptr(commit), _ptr(o), _stream(stream)),
           "hb_block_attend_commit_s16")
    return o


def hb_prefill_attend(cfg: Config, slot_idx, q, k, v, S_pool, Z_pool, W, gate_logits,
                      accumulate: bool = False, o=None, stream=None) -> torch.Tensor:
    """Prompts q/k/v [B, T, H, d] (T a multiple of L) processed block by
    block: block j attends against the state of blocks 0 .. j-1 (plus the
    slot's state when accumulate), then is committed. Returns o [B, T, H, d];
    the slots end up holding the whole prompt's state."""
    B = slot_idx.shape[0]
    H, d, f = cfg.num_heads, cfg.head_dim, cfg.feat_half
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    T = q.shape[1] if q.dim() == 4 else -1
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, cfg.torch_dtype, (B, T, H, d))
    num_slots = _check_state(cfg, S_pool, Z_pool)
    _check(W, "W", cfg.torch_dtype, (H, d, f))
    _check(gate_logits, "gate_logits", torch.float32, (H,))
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", cfg.torch_dtype, (B, T, H, d))
    lib = _lib.load()
    _raise(lib.hb_prefill_attend(ctypes.byref(cfg.c()), B, _ptr(slot_idx), _ptr(q), _ptr(k),
                                 _ptr(v), T, _ptr(S_pool), _ptr(Z_pool), num_slots, _ptr(W),
                                 _ptr(gate_logits), 1 if accumulate else 0, _ptr(o),
                                 _stream(stream)),
           "hb_prefill_attend")
    return o


def hb_block_attend_ex(cfg: Config, num_kv_heads: int, slot_idx, q, k, v, S_pool, Z_pool, Wq,
                       gate_logits, Wk=None, commit=None, o=None, stream=None) -> torch.Tensor:
    """Grouped-query heads and/or separate query and key maps: q [B, L, H, d],
    k/v [B, L, H_kv, d], states per key/value head, Wq [H, d, f],
    Wk [H_kv, d, f] (commits only). With ``commit``, requests with
    commit[b] != 0 then fold their block into their slot."""
    B = slot_idx.shape[0]
    H, d, f, L = cfg.num_heads, cfg.head_dim, cfg.feat_half, cfg.block_len
    Hkv = int(num_kv_heads)
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    _check(q, "q", cfg.torch_dtype, (B, L, H, d))
    _check(k, "k", cfg.torch_dtype, (B, L, Hkv, d))
    _check(v, "v", cfg.torch_dtype, (B, L, Hkv, d))
    if S_pool.dim() != 4:
        raise ValueError("S_pool: expected [num_slots, H_kv, F, d]")
    num_slots = S_pool.shape[0]
    _check(S_pool, "S_pool", torch.float32, (num_slots, Hkv, cfg.F, d))
    _check(Z_pool, "Z_pool", torch.float32, (num_slots, Hkv, cfg.F))
    _check(Wq, "Wq", cfg.torch_dtype, (H, d, f))
    if Wk is not None:
        _check(Wk, "Wk", cfg.torch_dtype, (Hkv, d, f))
    if commit is not None:
        _check(commit, "commit", torch.int32, (B,))
        if Wk is None:
            raise ValueError("Wk: the key map is needed to commit")
    _check(gate_logits, "gate_logits", torch.float32, (H,))
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", cfg.torch_dtype, (B, L, H, d))
    lib = _lib.load()
    _raise(lib.hb_block_attend_ex(ctypes.byref(cfg.c()), Hkv, B, _ptr(slot_idx), _ptr(q), _ptr(k),
                                  _ptr(v), _ptr(S_pool), _ptr(Z_pool), num_slots, _ptr(Wq),
                                  _ptr(Wk), _ptr(gate_logits), _ptr(commit), _ptr(o),
                                  _stream(stream)), "hb_block_attend_ex")
    return o


def hb_prefill_attend_ex(cfg: Config, num_kv_heads: int, slot_idx, q, k, v, S_pool, Z_pool, Wq,
                         Wk, gate_logits, accumulate: bool = False, o=None,
                         stream=None) -> torch.Tensor:
    """hb_prefill_attend with grouped-query heads and/or separate maps:
    q [B, T, H, d], k/v [B, T, H_kv, d], states per key/value head."""
    B = slot_idx.shape[0]
    H, d, f = cfg.num_heads, cfg.head_dim, cfg.feat_half
    Hkv = int(num_kv_heads)
    T = q.shape[1] if q.dim() == 4 else -1
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    _check(q, "q", cfg.torch_dtype, (B, T, H, d))
    _check(k, "k", cfg.torch_dtype, (B, T, Hkv, d))
    _check(v, "v", cfg.torch_dtype, (B, T, Hkv, d))
    if S_pool.dim() != 4:
        raise ValueError("S_pool: expected [num_slots, H_kv, F, d]")
    num_slots = S_pool.shape[0]
    _check(S_pool, "S_pool", torch.float32, (num_slots, Hkv, cfg.F, d))
    _check(Z_pool, "Z_pool", torch.float32, (num_slots, Hkv, cfg.F))
    _check(Wq, "Wq", cfg.torch_dtype, (H, d, f))
    _check(Wk, "Wk", cfg.torch_dtype, (Hkv, d, f))
    _check(gate_logits, "gate_logits", torch.float32, (H,))
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", cfg.torch_dtype, (B, T, H, d))
    lib = _lib.load()
    _raise(lib.hb_prefill_attend_ex(ctypes.byref(cfg.c()), Hkv, B, _ptr(slot_idx), _ptr(q),
                                    _ptr(k), _ptr(v), T, _ptr(S_pool), _ptr(Z_pool), num_slots,
                                    _ptr(Wq), _ptr(Wk), _ptr(gate_logits),
                                    int(bool(accumulate)), _ptr(o), _stream(stream)),
           "hb_prefill_attend_ex")
    return o


def hb_commit_block(cfg: Config, slot_idx, k, v, W, S_pool, Z_pool, stream=None) -> None:
    """S += sum_t phi(k_t) v_t^T, Z += sum_t phi(k_t) for each listed slot."""
    B = slot_idx.shape[0]
    H, d, f, L = cfg.num_heads, cfg.head_dim, cfg.feat_half, cfg.block_len
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    _check(k, "k", cfg.torch_dtype, (B, L, H, d))
    _check(v, "v", cfg.torch_dtype, (B, L, H, d))
    _check(W, "W", cfg.torch_dtype, (H, d, f))
    num_slots = _check_state(cfg, S_pool, Z_pool)
    lib = _lib.load()
    _raise(lib.hb_commit_block(ctypes.byref(cfg.c()), B, _ptr(slot_idx), _ptr(k), _ptr(v),
                               _ptr(W), _ptr(S_pool), _ptr(Z_pool), num_slots, _stream(stream)),
           "hb_commit_block")


def hb_prefill_workspace_size(cfg: Config, batch: int, max_seqlen: int) -> int:
    return int(_lib.load().hb_prefill_workspace_size(ctypes.byref(cfg.c()), batch, max_seqlen))


def hb_prefill_state(cfg: Config, slot_idx, k, v, cu_seqlens, max_seqlen: int, W, S_pool,
                     Z_pool, accumulate: bool = False, workspace=None, stream=None) -> None:
    """Ingest packed prompts k/v [total, H, d] (request b owns rows
    cu_seqlens[b]:cu_seqlens[b+1]) into the listed slots."""
    B = slot_idx.shape[0]
    H, d, f = cfg.num_heads, cfg.head_dim, cfg.feat_half
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    _check(cu_seqlens, "cu_seqlens", torch.int64, (B + 1,))
    total = k.shape[0]
    _check(k, "k", cfg.torch_dtype, (total, H, d))
    _check(v, "v", cfg.torch_dtype, (total, H, d))
    _check(W, "W", cfg.torch_dtype, (H, d, f))
    num_slots = _check_state(cfg, S_pool, Z_pool)
    need = hb_prefill_workspace_size(cfg, B, max_seqlen)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=k.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = _lib.load()
    _raise(lib.hb_prefill_state(ctypes.byref(cfg.c()), B, _ptr(slot_idx),
                                _ptr(k) if total else None, _ptr(v) if total else None,
                                total, _ptr(cu_seqlens), max_seqlen, _ptr(W), _ptr(S_pool),
                                _ptr(Z_pool), num_slots, int(bool(accumulate)), _ptr(workspace),
                                ws_bytes, _stream(stream)), "hb_prefill_state")


def hb_prefill_state_noalloc(cfg: Config, slot_idx, k, v, cu_seqlens, max_seqlen: int, W,
                             S_pool, Z_pool, accumulate: bool = False, stream=None) -> None:
    """hb_prefill_state without a workspace, for callers that cannot allocate
    device memory: the split partial sums go to the library's fixed scratch
    array (HB_PREFILL_NOALLOC_SCRATCH_BYTES). Calls that overlap on the GPU
    share that array and race; a shape that needs more scratch is rejected."""
    B = slot_idx.shape[0]
    H, d, f = cfg.num_heads, cfg.head_dim, cfg.feat_half
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    _check(cu_seqlens, "cu_seqlens", torch.int64, (B + 1,))
    total = k.shape[0]
    _check(k, "k", cfg.torch_dtype, (total, H, d))
    _check(v, "v", cfg.torch_dtype, (total, H, d))
    _check(W, "W", cfg.torch_dtype, (H, d, f))
    num_slots = _check_state(cfg, S_pool, Z_pool)
    lib = _lib.load()
    _raise(lib.hb_prefill_state_noalloc(ctypes.byref(cfg.c()), B, _ptr(slot_idx),
                                        _ptr(k) if total else None, _ptr(v) if total else None,
                                        total, _ptr(cu_seqlens), max_seqlen, _ptr(W),
                                        _ptr(S_pool), _ptr(Z_pool), num_slots,
                                        int(bool(accumulate)), _stream(stream)),
           "hb_prefill_state_noalloc")


def hb_state_zero(cfg: Config, slot_idx, S_pool, Z_pool, stream=None) -> None:
    B = slot_idx.shape[0]
    _check(slot_idx, "slot_idx", torch.int32, (B,))
    num_slots = _check_state(cfg, S_pool, Z_pool)
    lib = _lib.load()
    _raise(lib.hb_state_zero(ctypes.byref(cfg.c()), B, _ptr(slot_idx), _ptr(S_pool),
                             _ptr(Z_pool), num_slots, _stream(stream)), "hb_state_zero")


def hb_state_copy(cfg: Config, src_slot, dst_slot, S_pool, Z_pool, stream=None) -> None:
    """Copies the states of slots src_slot[b] to slots dst_slot[b] (distinct
    destinations, none of them also a source in the same call)."""
    B = src_slot.shape[0]
    _check(src_slot, "src_slot", torch.int32, (B,))
    _check(dst_slot, "dst_slot", torch.int32, (B,))
    num_slots = _check_state(cfg, S_pool, Z_pool)
    lib = _lib.load()
    _raise(lib.hb_state_copy(ctypes.byref(cfg.c()), B, _ptr(src_slot), _ptr(dst_slot),
                             _ptr(S_pool), _ptr(Z_pool), num_slots, _stream(stream)),
           "hb_state_copy")


def hb_softmax_kv_workspace_size(cfg: Config, batch: int, max_prefix: int) -> int:
    return int(_lib.load().hb_softmax_kv_workspace_size(ctypes.byref(cfg.c()), batch, max_prefix))


def hb_softmax_kv_attend(cfg: Config, k_cache, v_cache, cu_prefix, max_prefix: int, q, k, v,
                         o=None, workspace=None, stream=None) -> torch.Tensor:
    """Comparison path: full-prefix softmax attention of the active block over a
    packed KV cache [total_prefix, H, d] followed by the block itself."""
    B = q.shape[0]
    H, d, L = cfg.num_heads, cfg.head_dim, cfg.block_len
    _check(cu_prefix, "cu_prefix", torch.int64, (B + 1,))
    total = k_cache.shape[0]
    _check(k_cache, "k_cache", cfg.torch_dtype, (total, H, d))
    _check(v_cache, "v_cache", cfg.torch_dtype, (total, H, d))
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, cfg.torch_dtype, (B, L, H, d))
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", cfg.torch_dtype, (B, L, H, d))
    need = hb_softmax_kv_workspace_size(cfg, B, max_prefix)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = _lib.load()
    _raise(lib.hb_softmax_kv_attend(ctypes.byref(cfg.c()), B, _ptr(k_cache) if total else None,
                                    _ptr(v_cache) if total else None, total, _ptr(cu_prefix),
                                    max_prefix, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                    _ptr(workspace), ws_bytes, _stream(stream)),
           "hb_softmax_kv_attend")
    return o


def hb_softmax_kv_attend_paged(cfg: Config, k_pages, v_pages, page_table, prefix_len,
                               max_prefix: int, q, k, v, o=None, workspace=None,
                               stream=None) -> torch.Tensor:
    """Comparison path over a paged KV cache: k_pages/v_pages [num_pages,
    page_tokens, H, d] shared by all requests, page_table [B, max_pages] int32
    (request b's pages in token order), prefix_len [B] int32 cached tokens."""
    B = q.shape[0]
    H, d, L = cfg.num_heads, cfg.head_dim, cfg.block_len
    num_pages, page_tokens = k_pages.shape[0], k_pages.shape[1]
    _check(k_pages, "k_pages", cfg.torch_dtype, (num_pages, page_tokens, H, d))
    _check(v_pages, "v_pages", cfg.torch_dtype, (num_pages, page_tokens, H, d))
    max_pages = page_table.shape[1] if page_table.dim() == 2 else -1
    _check(page_table, "page_table", torch.int32, (B, max_pages))
    _check(prefix_len, "prefix_len", torch.int32, (B,))
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, cfg.torch_dtype, (B, L, H, d))
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", cfg.torch_dtype, (B, L, H, d))
    need = hb_softmax_kv_workspace_size(cfg, B, max_prefix)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = _lib.load()
    _raise(lib.hb_softmax_kv_attend_paged(
        ctypes.byref(cfg.c()), B, _ptr(k_pages) if num_pages else None,
        _ptr(v_pages) if num_pages else None, num_pages, page_tokens,
        _ptr(page_table) if max_pages else None, max_pages, _ptr(prefix_len), max_prefix,
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(workspace), ws_bytes, _stream(stream)),
        "hb_softmax_kv_attend_paged")
    return o


def hb_set_wait_limit(cycles: int) -> None:
    """Test hook: the attend kernels' pipeline waits give up after ``cycles``
    SM clocks (0 restores the default); process-wide."""
    _raise(_lib.load().hb_set_wait_limit(int(cycles)), "hb_set_wait_limit")


def hb_get_device_status(stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device status code."""
    return int(_lib.load().hb_get_device_status(_stream(stream)))


def hb_status_string(status: int) -> str:
    return _lib.load().hb_status_string(status).decode()
