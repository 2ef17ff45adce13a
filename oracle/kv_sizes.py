"""KV-cache memory arithmetic (test infrastructure only).

* "KV Cache는 왜 LLM 서빙의 핵심인가", section "KV Cache: O(T²)를 O(T)로"
  (trade-off box) and section "메모리 공식과 GQA의 동기": one request holds
  M_KV = 2 * L * T * d_cache * b bytes (K and V, L layers, T tokens, d_cache
  cached values per token per layer, b bytes per value); with GQA the cached
  width is d_h * n_kv, a saving of n_h / n_kv.
* "LLM 서빙과 KV Cache, VLLM", section "KV Cache의 크기 계산 (naive)": the
  same count per token, 2 * layers * hidden * 2 bytes for FP16.
"""


def kv_bytes(L, T, d_cache, b):
    """M_KV = 2 * L * T * d_cache * b."""
    return 2 * L * T * d_cache * b


def kv_bytes_gqa(L, T, d_h, n_kv, b):
    """M_KV^GQA = 2 * L * T * (d_h * n_kv) * b."""
    return 2 * L * T * (d_h * n_kv) * b


def kv_bytes_per_token(L, hidden, b):
    """Bytes of K and V one token adds across L layers (MHA, d_cache = hidden)."""
    return kv_bytes(L, 1, hidden, b)
