"""Launch-shape determinism (page qkv_front, module docstring: no atomics, no
global scratch, the result depends on the launch shape only; ring_stages:
the ring depth does not change the result)."""
import numpy as np
import pytest
import torch

from kv_insert_gb300 import qkv_front as qf
from kv_insert_gb300 import workloads as wl

from _parity import assert_cache, assert_values, device_inputs, run_device, run_oracle

pytestmark = pytest.mark.gpu

# ring depths and K splits the GPU tests launch; tests/test_boundary.py checks
# on the CPU that the library accepts each of them
RING_DEPTHS = (2, 3, 4, 5)
SPLIT_CASES = [
    ("m8_nkv8_n9216", (1, 2, 4)),
    ("m1_nkv1_n1152", (1, 2, 4, 8, 16)),
    ("m16_nkv8_n9216_consecutive", (1, 2, 4, 8)),
]


def split_stages(splits):
    return 2 if splits == 16 else 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    qf.status()


def _fresh(inp):
    return device_inputs(inp)


@pytest.mark.parametrize("name", ["m8_nkv8_n9216", "m1_nkv1_n1152", "sweep_m13_nkv8_n9216"])
def test_repeat_runs_bitwise_equal(name):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    outs, caches = [], []
    for _ in range(3):
        g = _fresh(inp)
        outs.append(run_device(g))
        caches.append(g["kv_cache"])
    for o, c in zip(outs[1:], caches[1:]):
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
        assert torch.equal(c.view(torch.int16), caches[0].view(torch.int16))


ENGINES = [qf.CONSUMER_MMA_SYNC, qf.CONSUMER_TCGEN05]


@pytest.mark.parametrize("consumer", ENGINES, ids=["mma_sync", "tcgen05"])
@pytest.mark.parametrize("name,splits", [("m8_nkv8_n9216", 1), ("m16_nkv8_n9216_consecutive", 2),
                                         ("m1_nkv1_n1152", 8)])
def test_ring_depth_does_not_change_result(name, splits, consumer):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    ref = None
    for stages in RING_DEPTHS:
        g = _fresh(inp)
        out = run_device(g, splits=splits, stages=stages, consumer=consumer)
        if ref is None:
            ref = out
        else:
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), stages


@pytest.mark.parametrize("consumer", ENGINES, ids=["mma_sync", "tcgen05"])
@pytest.mark.parametrize("name,splits_list", SPLIT_CASES)
def test_every_k_split_matches_oracle(name, splits_list, consumer):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    out_ref, cache_ref, err = run_oracle(inp, w.num_kv_heads)
    assert err == 0
    for splits in splits_list:
        g = _fresh(inp)
        out = run_device(g, splits=splits, stages=split_stages(splits), consumer=consumer)
        assert qf.status() == 0
        out_bits = wl.bits(out.cpu())
        assert_values(out_bits, out_ref, what=f"out at splits={splits}")
        assert_cache(inp, w.num_kv_heads, g["kv_cache"], out_bits, cache_ref)
        again = run_device(_fresh(inp), splits=splits, stages=3, consumer=consumer)
        assert torch.equal(again.view(torch.int16), out.view(torch.int16))


@pytest.mark.parametrize("kb", [1, 2, 4])
def test_every_stage_size_matches_oracle(kb):
    w = wl.WORKLOADS["m16_nkv8_n9216_consecutive"]
    inp = wl.make_inputs(w)
    out_ref, cache_ref, err = run_oracle(inp, w.num_kv_heads)
    for consumer in ENGINES:
        g = _fresh(inp)
        out = run_device(g, splits=1, stages=3, kb=kb, consumer=consumer)
        assert qf.status() == 0
        out_bits = wl.bits(out.cpu())
        assert_values(out_bits, out_ref, what=f"out at kb={kb}, consumer={consumer}")
        assert_cache(inp, w.num_kv_heads, g["kv_cache"], out_bits, cache_ref)
