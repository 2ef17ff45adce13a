"""Oracle: a plain, slow, CPU restatement of what the paged decode path computes.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
CUDA library never imports, links or calls it, and it shares no code with the
CUDA library: no kernels, headers, helpers, tables or constant generators.

Arithmetic is float64 unless a step is defined in another precision (the INT4
quantizer follows a stated float32 / float16 op sequence so that its codes are
bit-exact by construction).

Sources (web pages; cited by title and section in every function):

* "KV 캐시 시스템 (KV Cache System)" — TensorRT-LLM KV cache wiki page
  (sections "MQA / GQA", "요청 간 재사용", "보존 정책", "제한된 어텐션 윈도우
  크기", "호스트 메모리로의 오프로딩", "어텐션 윈도우 크기").
* "LLM 서빙과 KV Cache, VLLM" — velog post (sections "KV Cache의 크기 계산
  (naive)", "VLLM", "PagedAttention").
* "KV Cache는 왜 LLM 서빙의 핵심인가" — iq-blog chapter 2 (sections
  "KV Cache: O(T²)를 O(T)로" with its decode-step listing, "메모리 공식과
  GQA의 동기" with the M_KV and M_KV^GQA equations, "KVQuant: 마지막 4배"
  with the quantization equation).
* "Research Paper Review : CACHE BLEND, Fast Large Language Model Serving for
  RAG with Cached Knowledge Fusion" — tistory review (section "Background",
  full KV reuse with RoPE re-rotation; sections "Methods" and "System Design", KV
  deviation, token selection and the recompute ratio).

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` (closed forms printed on the pages, invariants the
pages state, brute force on tiny inputs, textbook special cases).  None is
"parity unpinned".
"""
from .rounding import round_bf16, round_fp16_from_f32
from .paged_attention import (kv_append, gather_sequence, paged_decode_attention,
                              attention_weights, window_start, layer_windows)
from .kv_sizes import kv_bytes, kv_bytes_gqa, kv_bytes_per_token
from .int4 import (quantize_group, quantize_groups, pack_codes, unpack_codes, Int4Cache,
                   paged_decode_attention_int4)
from .rope import rope_shift_k, rotate
from .brute import attention_loops
from .block_manager import BlockManager, OutOfBlocks, apply_copies
from . import cacheblend

__all__ = [
    "round_bf16", "round_fp16_from_f32", "kv_append", "gather_sequence",
    "paged_decode_attention", "attention_weights", "kv_bytes", "kv_bytes_gqa",
    "kv_bytes_per_token", "quantize_group", "quantize_groups", "pack_codes", "unpack_codes", "Int4Cache",
    "paged_decode_attention_int4", "rope_shift_k", "rotate", "attention_loops", "window_start",
    "layer_windows", "BlockManager", "OutOfBlocks", "apply_copies", "cacheblend",
]
