"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
the same seeded inputs, at the full sizes of every workload.

Bar: BF16 values within |d| <= 2e-2 + 1e-2 |oracle|; cache placement exact
(only named slots change and each holds its token's k / v head bits); with
integer-valued inputs the projection is exact in any summation order, so the
v and gate columns must match the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

from kv_insert_gb300 import qkv_front as qf
from kv_insert_gb300 import workloads as wl

from _parity import (assert_cache, assert_values, check_workload, device_inputs, run_device,
                     run_oracle)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    qf.status()   # clear any bit left by an earlier module


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_workload_matches_oracle(name):
    check_workload(wl.WORKLOADS[name])


ENGINES = [qf.CONSUMER_MMA_SYNC, qf.CONSUMER_TCGEN05]


@pytest.mark.parametrize("consumer", ENGINES, ids=["mma_sync", "tcgen05"])
@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_each_engine_matches_oracle(name, consumer):
    """Both contraction engines at the library's split and ring depth."""
    w = wl.WORKLOADS[name]
    v = qf.variant_full(w.N, w.M)
    check_workload(w, splits=v["splits"], stages=v["stages"], kb=v["kb"], consumer=consumer)


def _vg_cols(nkv):
    q_width = 8 * nkv * 64
    return slice(q_width + nkv * 64, None)   # v then gate heads


@pytest.mark.parametrize("name", ["m1_nkv1_n1152", "m8_nkv8_n9216", "m16_nkv8_n9216_consecutive",
                                  "sweep_m13_nkv8_n9216", "m8_nkv16_n18432"])
@pytest.mark.parametrize("consumer", ENGINES, ids=["mma_sync", "tcgen05"])
def test_integer_inputs_bit_exact_projection(name, consumer):
    w = wl.WORKLOADS[name]
    v = qf.variant_full(w.N, w.M)
    _, out_bits, out_ref = check_workload(w, integer_valued=True, splits=v["splits"],
                                          stages=v["stages"], kb=v["kb"], consumer=consumer)
    vg = _vg_cols(w.num_kv_heads)
    assert np.array_equal(out_bits[:, vg], out_ref[:, vg])


@pytest.mark.parametrize("consumer", ENGINES, ids=["mma_sync", "tcgen05"])
@pytest.mark.parametrize("M", list(range(1, 17)))
def test_every_token_count_one_kv_head(M, consumer):
    """Every M from 1 to 16 (ragged 8-token tiles) at N = 1152."""
    w = wl.Workload(f"m{M}_nkv1", M=M, num_kv_heads=1, max_pos=4096, num_pages=8, seed=2000 + M)
    v = qf.variant_full(w.N, w.M)
    check_workload(w, splits=v["splits"], stages=v["stages"], kb=v["kb"], consumer=consumer)


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_resident_engine_every_token_count(M):
    """The library's choice at N = 1152 (K split 8 ways): the resident engine
    (the whole W share on chip before the wait, partials pushed to the owner
    rank), every M from 1 to 16, against the oracle; a second run gives the
    same bits in out and in the cache."""
    w = wl.Workload(f"r{M}_nkv1", M=M, num_kv_heads=1, max_pos=4096, num_pages=8, seed=2300 + M)
    v = qf.variant_full(w.N, w.M)
    assert (v["consumer"], v["splits"], v["kb"], v["stages"]) == ("resident", 8, 4, 4)
    inp, out_bits, _ = check_workload(w)
    g = device_inputs(inp)
    again = run_device(g)
    assert np.array_equal(wl.bits(again.cpu()), out_bits)
    g2 = device_inputs(inp)
    run_device(g2, splits=8, stages=4, kb=4, consumer=qf.CONSUMER_RESIDENT)
    assert torch.equal(g2["kv_cache"].view(torch.int16), g["kv_cache"].view(torch.int16))


@pytest.mark.parametrize("M", [1, 8, 9, 16])
def test_resident_engine_integer_inputs_bit_exact(M):
    """Integer-valued x and W: every partial sum is exact, so the resident
    engine's own k order inside its register stages cannot change a bit of
    the v and gate columns."""
    w = wl.Workload(f"ri{M}_nkv1", M=M, num_kv_heads=1, max_pos=4096, num_pages=8, seed=2400 + M)
    _, out_bits, out_ref = check_workload(w, integer_valued=True)
    vg = _vg_cols(1)
    assert np.array_equal(out_bits[:, vg], out_ref[:, vg])


def test_resident_engine_index_rules():
    """Negative, past-the-cache slots and a position past the table on the
    resident engine: flagged, skipped, nothing written outside a cache view."""
    w = wl.Workload("rbad", M=7, num_kv_heads=1, max_pos=512, num_pages=4, seed=2501)
    inp = wl.make_inputs(w)
    inp["slots"][1] = -1
    inp["slots"][4] = w.num_pages * 16 + 3
    inp["positions"][6] = w.max_pos
    g = device_inputs(inp)
    parent = torch.zeros(2 * w.num_pages, 1, 16, 128, dtype=torch.bfloat16, device="cuda:0")
    parent[: w.num_pages].copy_(g["kv_cache"])
    g["kv_cache"] = parent[: w.num_pages]
    sentinel = torch.full((w.M, w.N), 3.0, dtype=torch.bfloat16)
    out = run_device(g, out=sentinel.to("cuda:0"))
    st = qf.status()
    assert int(parent[w.num_pages:].view(torch.int16).abs().sum()) == 0, "insert past the cache"
    out_bits = wl.bits(out.cpu())
    out_ref, cache_ref, err = run_oracle(inp, w.num_kv_heads, out_bits=wl.bits(sentinel))
    assert err == 3
    assert np.array_equal(out_bits[6, : 9 * 64], out_ref[6, : 9 * 64])   # untouched sentinel
    assert_values(out_bits, out_ref)
    assert_cache(inp, w.num_kv_heads, g["kv_cache"], out_bits, cache_ref)
    assert st == qf.STATUS_BAD_SLOT | qf.STATUS_BAD_POSITION, st


@pytest.mark.parametrize("nkv", [2, 3, 4])
def test_other_kv_head_counts(nkv):
    w = wl.Workload(f"m5_nkv{nkv}", M=5, num_kv_heads=nkv, max_pos=8192, num_pages=64,
                    seed=2100 + nkv)
    check_workload(w)


@pytest.mark.parametrize("nkv,M", [(24, 9), (64, 2)])
def test_many_kv_heads(nkv, M):
    """Up to the most KV heads the front accepts (64: N = 73728, 1152 heads,
    several waves of CTAs), with a ragged second token tile at M = 9."""
    w = wl.Workload(f"m{M}_nkv{nkv}", M=M, num_kv_heads=nkv, max_pos=4096, num_pages=64,
                    seed=2150 + nkv)
    check_workload(w)


def test_negative_slot_inserts_nothing():
    w = wl.Workload("pad", M=6, num_kv_heads=2, max_pos=1024, num_pages=16, seed=2201)
    inp = wl.make_inputs(w)
    inp["slots"][2] = -1
    g = device_inputs(inp)
    out = run_device(g)
    assert qf.status() == 0
    out_bits = wl.bits(out.cpu())
    out_ref, cache_ref, err = run_oracle(inp, w.num_kv_heads)
    assert err == 0
    assert_values(out_bits, out_ref)
    assert_cache(inp, w.num_kv_heads, g["kv_cache"], out_bits, cache_ref)


def test_out_of_range_slot_and_position_are_flagged_not_written():
    """Checked in the kernel: a slot past the cache and a position past the
    table raise status bits; that token's insert (and for the position, its
    q and k heads) is skipped.  The cache is a view of the first pages of a
    larger buffer, so a wrong insert would land in memory the test owns and
    is seen in the pages past the view."""
    w = wl.Workload("bad", M=4, num_kv_heads=1, max_pos=512, num_pages=4, seed=2202)
    inp = wl.make_inputs(w)
    inp["slots"][1] = w.num_pages * 16 + 5
    inp["positions"][3] = w.max_pos + 7
    g = device_inputs(inp)
    parent = torch.zeros(2 * w.num_pages, 1, 16, 128, dtype=torch.bfloat16, device="cuda:0")
    parent[: w.num_pages].copy_(g["kv_cache"])
    g["kv_cache"] = parent[: w.num_pages]
    assert g["kv_cache"].is_contiguous()
    sentinel = torch.full((w.M, w.N), 3.0, dtype=torch.bfloat16)
    out = run_device(g, out=sentinel.to("cuda:0"))
    st = qf.status()
    assert int(parent[w.num_pages:].view(torch.int16).abs().sum()) == 0, "insert past the cache"
    out_bits = wl.bits(out.cpu())
    out_ref, cache_ref, err = run_oracle(inp, w.num_kv_heads, out_bits=wl.bits(sentinel))
    assert err == 3
    assert np.array_equal(out_bits[3, : 9 * 64], out_ref[3, : 9 * 64])   # untouched sentinel
    assert_values(out_bits, out_ref)
    assert_cache(inp, w.num_kv_heads, g["kv_cache"], out_bits, cache_ref)
    assert st == qf.STATUS_BAD_SLOT | qf.STATUS_BAD_POSITION, st


@pytest.mark.parametrize("which", ["slot", "position"])
def test_each_bad_index_alone_is_flagged(which):
    w = wl.Workload("bad1", M=3, num_kv_heads=2, max_pos=256, num_pages=2, seed=2203)
    inp = wl.make_inputs(w)
    if which == "slot":
        inp["slots"][0] = w.num_pages * 16
    else:
        inp["positions"][2] = -5
    g = device_inputs(inp)
    parent = torch.zeros(2 * w.num_pages, 2, 16, 128, dtype=torch.bfloat16, device="cuda:0")
    parent[: w.num_pages].copy_(g["kv_cache"])
    g["kv_cache"] = parent[: w.num_pages]
    run_device(g)
    st = qf.status()
    assert int(parent[w.num_pages:].view(torch.int16).abs().sum()) == 0, "insert past the cache"
    want = qf.STATUS_BAD_SLOT if which == "slot" else qf.STATUS_BAD_POSITION
    assert st == want, st


def test_zero_tokens_launches_nothing():
    w = wl.WORKLOADS["m1_nkv1_n1152"]
    inp = wl.make_inputs(w)
    g = device_inputs(inp)
    before = g["kv_cache"].clone()
    out = torch.empty(0, w.N, dtype=torch.bfloat16, device="cuda:0")
    qf.qkv_front(g["x"][:0], g["W"], g["positions"][:0], g["slots"][:0], g["cos_sin"],
                 g["kv_cache"], out)
    torch.cuda.synchronize()
    assert torch.equal(before, g["kv_cache"])


@pytest.mark.parametrize("name", ["m8_nkv8_n9216", "sweep_m13_nkv8_n9216"])
def test_from_host_entry_matches_device_call(name):
    """qkv_front_from_host (host x / positions / slots in, out back to host)
    gives the device call's bits, in out and in the cache."""
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    g = device_inputs(inp)
    out_dev = run_device(g)
    cache_dev = g["kv_cache"].clone()
    g2 = device_inputs(inp)
    xh, ph, sh = inp["x"].pin_memory(), inp["positions"].pin_memory(), inp["slots"].pin_memory()
    oh = torch.zeros(w.M, w.N, dtype=torch.bfloat16).pin_memory()
    staging = torch.empty(qf.staging_bytes(w.M, w.N), dtype=torch.uint8, device="cuda:0")
    for _ in range(2):
        qf.qkv_front_from_host(xh, ph, sh, oh, g2["W"], g2["cos_sin"], g2["kv_cache"], staging)
        torch.cuda.synchronize()
        assert qf.status() == 0
        assert torch.equal(oh.view(torch.int16), out_dev.cpu().view(torch.int16))
        assert torch.equal(g2["kv_cache"].view(torch.int16), cache_dev.view(torch.int16))


@pytest.mark.parametrize("pinned_in,pinned_out", [(False, False), (True, False), (False, True)])
def test_from_host_pageable_buffers_take_the_copy_path(pinned_in, pinned_out):
    """Pinned host buffers are read and written by the kernels directly;
    pageable ones are copied on the stream.  Every mix gives the device
    call's bits."""
    w = wl.WORKLOADS["m8_nkv8_n9216"]
    inp = wl.make_inputs(w)
    g = device_inputs(inp)
    out_dev = run_device(g)
    cache_dev = g["kv_cache"].clone()
    g2 = device_inputs(inp)
    pin = (lambda t: t.pin_memory()) if pinned_in else (lambda t: t.clone())
    xh, ph, sh = pin(inp["x"]), pin(inp["positions"]), pin(inp["slots"])
    oh = torch.zeros(w.M, w.N, dtype=torch.bfloat16)
    if pinned_out:
        oh = oh.pin_memory()
    staging = torch.empty(qf.staging_bytes(w.M, w.N), dtype=torch.uint8, device="cuda:0")
    qf.qkv_front_from_host(xh, ph, sh, oh, g2["W"], g2["cos_sin"], g2["kv_cache"], staging)
    torch.cuda.synchronize()
    assert qf.status() == 0
    assert torch.equal(oh.view(torch.int16), out_dev.cpu().view(torch.int16))
    assert torch.equal(g2["kv_cache"].view(torch.int16), cache_dev.view(torch.int16))


def test_page_helper_names():
    """The pages' helper names on this device: k_split, ring_stages,
    sm100_family, compile_qkv_front."""
    assert qf.sm100_family()
    assert qf.k_split(9216) == 1 and qf.k_split(1152) == 8
    assert qf.ring_stages(9216, 8) == qf.variant_full(9216, 8)["stages"] >= 2
    qf.compile_qkv_front(9216, 8)
