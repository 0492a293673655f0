"""The memory-capacity helper against byte counts worked out by hand (CPU)."""

import pytest

from linear_attention_diffusion_feature_b300 import capacity


def test_kv_cache_bytes_by_hand():
    # one 32-token page of one layer: 32 tokens x (k + v) x 16 heads x 128 x 2 B
    assert capacity.kv_cache_bytes(1, 1) == 32 * 2 * 16 * 128 * 2 == 262144
    assert capacity.kv_cache_bytes(32, 1) == 262144
    assert capacity.kv_cache_bytes(33, 1) == 2 * 262144
    assert capacity.kv_cache_bytes(0, 20) == 0
    # 3,072 tokens in 20 layers: 96 pages x 256 KiB x 20
    assert capacity.kv_cache_bytes(3072, 20) == 96 * 262144 * 20 == 503316480


def test_state_bytes_by_hand():
    # S 128 x 128 and Z 128 fp32 per head, 16 heads
    assert capacity.state_bytes(1) == 16 * (128 * 128 + 128) * 4 == 1056768
    assert capacity.state_bytes(6) == 6 * 1056768


def test_hybrid_mix_and_concurrency():
    teacher = capacity.request_bytes(3072, 20, 0)
    hybrid = capacity.request_bytes(3072, 14, 6)
    assert teacher == 503316480
    assert hybrid == 14 * 96 * 262144 + 6 * 1056768 == 358662144
    budget = 100 * 2 ** 30
    assert capacity.max_requests(budget, 3072, 20, 0) == budget // teacher == 213
    assert capacity.max_requests(budget, 3072, 14, 6) == budget // hybrid == 299


def test_break_even():
    # 1,056,768 B of state = 129 tokens of one layer's KV; with 32-token
    # pages the cache first exceeds it at 5 pages
    t = capacity.break_even_tokens()
    assert t == 160
    assert capacity.kv_cache_bytes(t, 1) > capacity.state_bytes(1) >= \
        capacity.kv_cache_bytes(t - 32, 1)


def test_rejects_bad_sizes():
    with pytest.raises(ValueError):
        capacity.kv_cache_bytes(-1, 1)
    with pytest.raises(ValueError):
        capacity.kv_cache_bytes(1, 1, page_tokens=0)
    with pytest.raises(ValueError):
        capacity.state_bytes(-1)
