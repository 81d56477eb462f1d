"""The predecessor kernel (layer_front) against the oracle, and the PDL chain
layer_front -> qkv_front: the front streams its weights before the
predecessor finishes, yet reads the predecessor's output only after it."""
import numpy as np
import pytest
import torch

import oracle
from kv_insert_gb300 import qkv_front as qf
from kv_insert_gb300 import workloads as wl

from _parity import assert_values

pytestmark = pytest.mark.gpu

H = 8192


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    qf.status()


@pytest.mark.parametrize("x_f32", [False, True], ids=["x_bf16", "x_fp32"])
@pytest.mark.parametrize("with_weight", [False, True], ids=["weightless", "weight"])
@pytest.mark.parametrize("rows", [1, 8, 16, 100])
def test_layer_front_matches_oracle(rows, x_f32, with_weight):
    g = torch.Generator().manual_seed(500 + rows)
    x = torch.randn(rows, H, generator=g) * 3
    x[rows // 2] *= 100.0                       # one loud row
    x = x if x_f32 else x.to(torch.bfloat16)
    w = (1.0 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16) if with_weight else None
    dev = "cuda:0"
    xd = x.to(dev)
    stream = torch.full((rows, H), float("nan"), device=dev)
    aux = torch.full((rows, H), float("nan"), device=dev)
    out = torch.empty(rows, H, dtype=torch.bfloat16, device=dev)
    qf.layer_front(xd, stream, out, aux=aux, weight=None if w is None else w.to(dev))
    torch.cuda.synchronize()
    xo = x.numpy() if x_f32 else wl.bits(x)
    s_ref, a_ref, o_ref = oracle.layer_front(xo, None if w is None else wl.bits(w), keep_aux=True)
    assert np.array_equal(stream.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(aux.cpu().numpy().view(np.uint32), a_ref.view(np.uint32))
    got = wl.bits(out.cpu())
    assert_values(got, o_ref, what="layer_front out")
    assert np.mean(got == o_ref) > 0.98


def test_layer_front_zero_rows_and_no_aux():
    dev = "cuda:0"
    x = torch.randn(4, H, device=dev).to(torch.bfloat16)
    stream = torch.zeros(4, H, device=dev)
    out = torch.zeros(4, H, dtype=torch.bfloat16, device=dev)
    qf.layer_front(x[:0], stream[:0], out[:0])
    torch.cuda.synchronize()
    assert not stream.any() and not out.float().any()
    qf.layer_front(x, stream, out)
    torch.cuda.synchronize()
    assert torch.equal(stream, x.float())


def _chain_inputs(name):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    lf = wl.make_layer_front_inputs(w)
    dev = "cuda:0"
    g = {k: v.to(dev) for k, v in inp.items()}
    g.update({k: v.to(dev) for k, v in lf.items()})
    g["stream"] = torch.empty(w.M, H, device=dev)
    g["x_attn"] = torch.empty(w.M, H, dtype=torch.bfloat16, device=dev)
    g["out"] = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    return w, inp, lf, g


def _chain(g, sync_between):
    qf.layer_front(g["x_embed"], g["stream"], g["x_attn"], weight=g["norm_weight"])
    if sync_between:
        torch.cuda.synchronize()
    qf.qkv_front(g["x_attn"], g["W"], g["positions"], g["slots"], g["cos_sin"], g["kv_cache"],
                 g["out"])
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["m8_nkv8_n9216", "m1_nkv1_n1152", "m16_nkv8_n9216_consecutive"])
def test_pdl_chain_equals_serialized_calls(name):
    """Back to back on one stream (the front starts during the predecessor)
    gives the same bits as the two calls with a device sync in between."""
    w, inp, lf, g1 = _chain_inputs(name)
    _chain(g1, sync_between=True)
    _, _, _, g2 = _chain_inputs(name)
    for _ in range(3):
        g2["out"].fill_(float("nan"))
        _chain(g2, sync_between=False)
        assert torch.equal(g2["out"].view(torch.int16), g1["out"].view(torch.int16))
        assert torch.equal(g2["x_attn"].view(torch.int16), g1["x_attn"].view(torch.int16))
    assert qf.status() == 0


def test_chain_without_pdl_gives_the_same_bits():
    w, inp, lf, g1 = _chain_inputs("m8_nkv8_n9216")
    _chain(g1, sync_between=False)
    _, _, _, g2 = _chain_inputs("m8_nkv8_n9216")
    qf.set_pdl(False)
    try:
        _chain(g2, sync_between=False)
    finally:
        qf.set_pdl(True)
    assert torch.equal(g2["out"].view(torch.int16), g1["out"].view(torch.int16))


def test_pdl_chain_in_a_graph_matches_oracle():
    """The chain captured in a CUDA graph (PDL edges kept) against the oracle
    chain: oracle layer_front, then the oracle front on its output."""
    w, inp, lf, g = _chain_inputs("m8_nkv8_n9216")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _chain(g, sync_between=False)       # warm (kernel attributes set)
    graph = torch.cuda.CUDAGraph()
    g["kv_cache"].copy_(inp["kv_cache"].to("cuda:0"))
    with torch.cuda.graph(graph, stream=s):
        qf.layer_front(g["x_embed"], g["stream"], g["x_attn"], weight=g["norm_weight"])
        qf.qkv_front(g["x_attn"], g["W"], g["positions"], g["slots"], g["cos_sin"], g["kv_cache"],
                     g["out"])
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    _, _, x_ref = oracle.layer_front(wl.bits(lf["x_embed"]), wl.bits(lf["norm_weight"]))
    cache = wl.bits(inp["kv_cache"]).copy()
    out_ref, err = oracle.qkv_front(x_ref, wl.bits(inp["W"]), inp["positions"].numpy(),
                                    inp["slots"].numpy(), inp["cos_sin"].numpy(), cache,
                                    w.num_kv_heads)
    assert err == 0
    assert_values(wl.bits(g["x_attn"].cpu()), x_ref, what="x_attn")
    assert_values(wl.bits(g["out"].cpu()), out_ref, what="front after the chain")
