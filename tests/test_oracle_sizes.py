"""Pins the oracle's cache-size arithmetic to the numbers the pages print."""
import os

import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_cache_sizes.txt")


def _rows():
    rows = {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, inputs, value, unit, tol, src = [x.strip() for x in line.split("|")]
            kv = dict(p.split("=") for p in inputs.split())
            rows[name] = (kv, float(value), unit, tol, src)
    return rows


ROWS = _rows()
UNIT = {"B": 1, "KiB": 1024, "GiB": 1024 ** 3, "GB": 1e9, "x": 1}


def _check(name, computed):
    kv, value, unit, tol, src = ROWS[name]
    got = computed / UNIT[unit]
    if tol == "exact":
        assert got == value, (name, got, value, src)
    else:
        assert abs(got - value) <= float(tol), (name, got, value, src)


def test_fixture_has_every_row():
    assert len(ROWS) == 9
    for _, (_, _, _, _, src) in ROWS.items():
        assert "section" in src


def test_per_token_naive():
    kv = ROWS["per_token_naive"][0]
    b = oracle.kv_bytes_per_token(int(kv["L"]), int(kv["hidden"]), int(kv["b"]))
    _check("per_token_naive", b)
    _check("per_token_naive_kb", b)


def test_llama7b_mha():
    kv = ROWS["llama7b_mha"][0]
    _check("llama7b_mha", oracle.kv_bytes(int(kv["L"]), int(kv["T"]), int(kv["d"]), int(kv["b"])))


def test_llama70b_mha():
    kv = ROWS["llama70b_mha"][0]
    one = oracle.kv_bytes(int(kv["L"]), int(kv["T"]), int(kv["d"]), int(kv["b"]))
    _check("llama70b_mha", one)
    _check("llama70b_mha_x100", 100 * one)


def test_llama70b_gqa():
    kv = ROWS["llama70b_gqa8"][0]
    g = oracle.kv_bytes_gqa(int(kv["L"]), int(kv["T"]), int(kv["d_h"]), int(kv["n_kv"]), int(kv["b"]))
    _check("llama70b_gqa8", g)
    # the saving against MHA is exactly n_h / n_kv (d = n_h * d_h)
    mha = oracle.kv_bytes(80, 2048, 64 * 128, 2)
    _check("gqa8_saving", mha / g)
    assert mha == 64 // 8 * g


def test_gqa_int4():
    kv = ROWS["llama70b_gqa8_int4"][0]
    g = oracle.kv_bytes_gqa(int(kv["L"]), int(kv["T"]), int(kv["d_h"]), int(kv["n_kv"]), float(kv["b"]))
    _check("llama70b_gqa8_int4", g)


def test_vllm_concurrency():
    kv = ROWS["vllm_concurrency"][0]
    _check("vllm_concurrency", int(kv["tokens"]) / int(kv["per_request"]))


@pytest.mark.parametrize("L,T,d,b", [(1, 1, 1, 1), (3, 5, 7, 2)])
def test_formula_counts_k_and_v(L, T, d, b):
    # one value of K and one of V per (layer, token, channel): brute count
    n = sum(1 for _ in range(2) for _ in range(L) for _ in range(T) for _ in range(d))
    assert oracle.kv_bytes(L, T, d, b) == n * b
