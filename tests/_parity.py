"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
the oracle on the same seeded inputs, and compare them."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from kv_insert_gb300 import qkv_front as qf
from kv_insert_gb300 import workloads as wl

# |gpu - oracle| <= TOL_ABS + TOL_REL * |oracle| on every BF16 output value
TOL_ABS = 2e-2
TOL_REL = 1e-2


def device_inputs(inp: dict, device="cuda:0") -> dict:
    return {k: v.to(device) for k, v in inp.items()}


def run_device(g: dict, splits=None, stages=None, out=None, kb=0, consumer=0):
    """One call through the C ABI: the library's own variant, or an explicit
    (splits, stages, kb, consumer) one."""
    M, N = g["x"].shape[0], g["W"].shape[0]
    if out is None:
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=g["x"].device)
    if splits is None:
        qf.qkv_front(g["x"], g["W"], g["positions"], g["slots"], g["cos_sin"], g["kv_cache"], out)
    else:
        qf.launch_variant(g["x"], g["W"], g["positions"], g["slots"], g["cos_sin"], g["kv_cache"],
                          out, splits, stages, kb=kb, consumer=consumer)
    torch.cuda.synchronize()
    return out


def run_oracle(inp: dict, nkv: int, out_bits=None):
    cache = wl.bits(inp["kv_cache"]).copy()
    out, err = oracle.qkv_front(wl.bits(inp["x"]), wl.bits(inp["W"]), inp["positions"].numpy(),
                                inp["slots"].numpy(), inp["cos_sin"].numpy(), cache, nkv,
                                out_bits=out_bits)
    return out, cache, err


def value_mismatch(got_bits: np.ndarray, ref_bits: np.ndarray):
    got = wl.from_bits(got_bits).float().numpy()
    ref = wl.from_bits(ref_bits).float().numpy()
    bad = ~(np.abs(got - ref) <= TOL_ABS + TOL_REL * np.abs(ref))
    return bad, got, ref


def assert_values(got_bits, ref_bits, what="out"):
    bad, got, ref = value_mismatch(got_bits, ref_bits)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} values outside tolerance; "
                             f"first {[(tuple(i), float(got[tuple(i)]), float(ref[tuple(i)])) for i in idx]}")


def assert_cache(inp: dict, nkv: int, cache_dev: torch.Tensor, out_bits: np.ndarray,
                 cache_ref: np.ndarray):
    """Placement is exact: only named slots change, and each holds exactly the
    k / v head bits of its token's out row; the values match the oracle's."""
    pre = wl.bits(inp["kv_cache"])
    cache = wl.bits(cache_dev.cpu())
    changed = np.argwhere((cache != pre).any(axis=(1, 3)))
    named = {}
    rows = inp["cos_sin"].shape[0]
    for t, (s, p) in enumerate(zip(inp["slots"].tolist(), inp["positions"].tolist())):
        if 0 <= s < pre.shape[0] * 16 and 0 <= p < rows:   # tokens that insert
            named[(s // 16, s % 16)] = t
    for pg, off in changed:
        assert (int(pg), int(off)) in named, f"slot {pg * 16 + off} written but named by no token"
    q_width, kv_width = 8 * nkv * 64, nkv * 64
    for (pg, off), t in named.items():
        for gkv in range(nkv):
            k = out_bits[t, q_width + gkv * 64: q_width + gkv * 64 + 64]
            v = out_bits[t, q_width + kv_width + gkv * 64: q_width + kv_width + gkv * 64 + 64]
            assert np.array_equal(cache[pg, gkv, off, :64], k), (t, gkv, "K")
            assert np.array_equal(cache[pg, gkv, off, 64:], v), (t, gkv, "V")
        assert_values(cache[pg, :, off, :], cache_ref[pg, :, off, :], what=f"cache slot {pg * 16 + off}")


def check_workload(w: wl.Workload, integer_valued=False, splits=None, stages=None, kb=0,
                   consumer=0):
    inp = wl.make_inputs(w, integer_valued=integer_valued)
    g = device_inputs(inp)
    out = run_device(g, splits, stages, kb=kb, consumer=consumer)
    assert qf.status() == 0
    out_bits = wl.bits(out.cpu())
    out_ref, cache_ref, err = run_oracle(inp, w.num_kv_heads)
    assert err == 0
    assert_values(out_bits, out_ref)
    assert_cache(inp, w.num_kv_heads, g["kv_cache"], out_bits, cache_ref)
    return inp, out_bits, out_ref
