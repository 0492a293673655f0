"""Device memory held per request by softmax layers (a paged KV cache that
grows with every token) and by linearized layers (a fixed-size state).

The pages attribute the hybrid model's higher concurrency to this difference:
the linearized layers keep a state whose size does not depend on the number
of committed tokens (gist.science technical summary, "Experimental Results",
"Throughput and Concurrency" bullets; pith.science referee report,
"Circularity Check", full rationale: S is 2F x d and Z is 2F, whatever the
number of committed tokens). This module sizes both, so that a
caller can split device memory between KV pages and state slots. It holds
byte counts only; nothing here touches a device.
"""

from __future__ import annotations


def kv_cache_bytes(tokens: int, layers: int, H: int = 16, d: int = 128,
                   page_tokens: int = 32, elem_bytes: int = 2) -> int:
    """k and v of ``tokens`` tokens in ``layers`` softmax layers, in whole
    pages of ``page_tokens`` tokens ([page_tokens, H, d] each for k and v)."""
    if tokens < 0 or layers < 0 or page_tokens <= 0:
        raise ValueError("tokens, layers >= 0 and page_tokens > 0 required")
    pages = -(-tokens // page_tokens)
    return layers * pages * page_tokens * 2 * H * d * elem_bytes


def state_bytes(layers: int, H: int = 16, f: int = 64, d: int = 128) -> int:
    """S [H, 2f, d] and Z [H, 2f] in fp32 for ``layers`` linearized layers."""
    if layers < 0:
        raise ValueError("layers >= 0 required")
    F = 2 * f
    return layers * H * (F * d + F) * 4


def request_bytes(tokens: int, softmax_layers: int, hybrid_layers: int, H: int = 16,
                  d: int = 128, f: int = 64, page_tokens: int = 32,
                  elem_bytes: int = 2) -> int:
    """Attention memory of one request after ``tokens`` tokens."""
    return (kv_cache_bytes(tokens, softmax_layers, H, d, page_tokens, elem_bytes)
            + state_bytes(hybrid_layers, H, f, d))


def max_requests(budget_bytes: int, tokens: int, softmax_layers: int, hybrid_layers: int,
                 **shape) -> int:
    """How many requests of ``tokens`` tokens fit in ``budget_bytes``."""
    per = request_bytes(tokens, softmax_layers, hybrid_layers, **shape)
    return budget_bytes // per if per > 0 else 0


def break_even_tokens(H: int = 16, d: int = 128, f: int = 64, page_tokens: int = 32,
                      elem_bytes: int = 2) -> int:
    """Smallest token count at which one layer's KV cache outgrows one
    layer's state."""
    s = state_bytes(1, H, f, d)
    t = 0
    while kv_cache_bytes(t, 1, H, d, page_tokens, elem_bytes) <= s:
        t += page_tokens
    return t
