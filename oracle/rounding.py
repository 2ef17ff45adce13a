"""Rounding to the storage formats of the cache (oracle side; test infrastructure only).

bfloat16 keeps 8 significant bits and float32's exponent range; round to nearest,
ties to even, is the rounding the decode path's stores use.  The pages fix no
storage precision beyond "FP16" for the cache-size arithmetic ("LLM 서빙과 KV
Cache, VLLM", section "KV Cache의 크기 계산 (naive)"); bf16 storage is the
workload's choice and fp16 is the INT4 metadata's.
"""
import numpy as np


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even); returns float64.

    Direct rounding from float64 (no float32 intermediate, so no double rounding).
    For |x| in the normal range the quantum is 2**(e-8) where x = m * 2**e with
    0.5 <= |m| < 1; below 2**-126 the quantum stays 2**-133 (bf16 subnormals).
    """
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    fin = np.isfinite(x) & (x != 0)
    xf = x[fin]
    _, e = np.frexp(xf)
    q = np.maximum(e, -125) - 8
    y = np.ldexp(np.rint(np.ldexp(xf, -q)), q)
    big = np.abs(y) >= 2.0 ** 128
    y[big] = np.copysign(np.inf, y[big])
    out[fin] = y
    return out


def round_fp16_from_f32(x) -> np.ndarray:
    """float32 -> float16, round to nearest even (numpy's conversion is correctly rounded)."""
    return np.asarray(x, dtype=np.float32).astype(np.float16)
