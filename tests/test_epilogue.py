"""The standalone epilogue (qknorm_rope_kv_insert, the unfused path's second
kernel) through the C ABI against the oracle: every token count from 1 to a
prefill chunk, values within tolerance, v and gate heads untouched bit for
bit, cache placement exact, index rules with status bits."""
import numpy as np
import pytest
import torch

import oracle
from kv_insert_gb300 import qkv_front as qf
from kv_insert_gb300 import workloads as wl

from _parity import assert_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    qf.status()


def run_both(inp, nkv, cache_parent_pages=None):
    dev = "cuda:0"
    g = {k: v.to(dev) for k, v in inp.items()}
    parent = None
    if cache_parent_pages:
        parent = torch.zeros(cache_parent_pages, *g["kv_cache"].shape[1:], dtype=torch.bfloat16,
                             device=dev)
        parent[: g["kv_cache"].shape[0]].copy_(g["kv_cache"])
        g["kv_cache"] = parent[: g["kv_cache"].shape[0]]
    qf.qknorm_rope_kv_insert(g["qkv"], g["positions"], g["slots"], g["cos_sin"], g["kv_cache"])
    torch.cuda.synchronize()
    st = qf.status()
    cache_ref = wl.bits(inp["kv_cache"]).copy()
    out_ref, err = oracle.qknorm_rope_kv_insert(wl.bits(inp["qkv"]), inp["positions"].numpy(),
                                                inp["slots"].numpy(), inp["cos_sin"].numpy(),
                                                cache_ref, nkv)
    return g, st, out_ref, cache_ref, err, parent


def check(inp, nkv, g, out_ref, cache_ref):
    got = wl.bits(g["qkv"].cpu())
    q_width, kv_width = 8 * nkv * 64, nkv * 64
    # v and gate heads: not touched
    assert np.array_equal(got[:, q_width + kv_width:], wl.bits(inp["qkv"])[:, q_width + kv_width:])
    assert_values(got, out_ref, what="qkv")
    same = np.mean(got == out_ref)
    assert same > 0.95, f"only {same:.3f} of values bit-equal to the oracle"
    pre = wl.bits(inp["kv_cache"])
    cache = wl.bits(g["kv_cache"].cpu())
    changed = {(int(a), int(b)) for a, b in np.argwhere((cache != pre).any(axis=(1, 3)))}
    rows = inp["cos_sin"].shape[0]
    named = {}
    for t, (s, p) in enumerate(zip(inp["slots"].tolist(), inp["positions"].tolist())):
        if 0 <= s < pre.shape[0] * 16 and 0 <= p < rows:
            named[(s // 16, s % 16)] = t
    assert changed <= set(named)
    for (pg, off), t in named.items():
        for gkv in range(nkv):
            assert np.array_equal(cache[pg, gkv, off, :64], got[t, q_width + gkv * 64:q_width + gkv * 64 + 64])
            assert np.array_equal(cache[pg, gkv, off, 64:],
                                  got[t, q_width + kv_width + gkv * 64:q_width + kv_width + gkv * 64 + 64])
    assert_values(cache[[k[0] for k in named], :, [k[1] for k in named], :],
                  cache_ref[[k[0] for k in named], :, [k[1] for k in named], :], what="cache")


@pytest.mark.parametrize("name", list(wl.EPI_WORKLOADS))
def test_epilogue_workloads_match_oracle(name):
    w = wl.EPI_WORKLOADS[name]
    inp = wl.make_epi_inputs(w)
    g, st, out_ref, cache_ref, err, _ = run_both(inp, w.num_kv_heads)
    assert st == 0 and err == 0
    check(inp, w.num_kv_heads, g, out_ref, cache_ref)


@pytest.mark.parametrize("T", [1, 2, 5, 16, 17, 31, 33, 64, 65, 255, 257])
def test_epilogue_token_counts(T):
    w = wl.EpiWorkload(f"t{T}", T=T, num_kv_heads=2, max_pos=2048, num_pages=64, seed=4000 + T)
    inp = wl.make_epi_inputs(w)
    g, st, out_ref, cache_ref, err, _ = run_both(inp, 2)
    assert st == 0 and err == 0
    check(inp, 2, g, out_ref, cache_ref)


@pytest.mark.parametrize("nkv", [4, 12, 16, 24, 64])
@pytest.mark.parametrize("T", [3, 37])
def test_epilogue_kv_head_counts(T, nkv):
    """Head counts on both sides of the two-items-per-token rule (16 KV heads
    and up) and the most the op accepts, at token counts far below the grid."""
    w = wl.EpiWorkload(f"t{T}_nkv{nkv}", T=T, num_kv_heads=nkv, max_pos=1024, num_pages=16,
                       seed=4200 + 100 * T + nkv)
    inp = wl.make_epi_inputs(w)
    g, st, out_ref, cache_ref, err, _ = run_both(inp, nkv)
    assert st == 0 and err == 0
    check(inp, nkv, g, out_ref, cache_ref)


@pytest.mark.parametrize("nkv", [1, 2, 4])
@pytest.mark.parametrize("T", [305, 1000, 2051])
def test_epilogue_four_cta_shape(T, nkv):
    """With 4 KV heads or fewer and more tokens than two CTAs per SM take,
    the kernel runs its four-CTA-per-SM shape (4 consumer warps): against
    the oracle, and bitwise on a repeat."""
    w = wl.EpiWorkload(f"s{T}_nkv{nkv}", T=T, num_kv_heads=nkv, max_pos=8192,
                       num_pages=(T + 15) // 16 + 64, seed=4400 + 10 * T + nkv)
    inp = wl.make_epi_inputs(w)
    g, st, out_ref, cache_ref, err, _ = run_both(inp, nkv)
    assert st == 0 and err == 0
    check(inp, nkv, g, out_ref, cache_ref)
    g2 = {k: v.to("cuda:0") for k, v in inp.items()}
    qf.qknorm_rope_kv_insert(g2["qkv"], g2["positions"], g2["slots"], g2["cos_sin"], g2["kv_cache"])
    torch.cuda.synchronize()
    assert torch.equal(g["qkv"].view(torch.int16), g2["qkv"].view(torch.int16))
    assert torch.equal(g["kv_cache"].view(torch.int16), g2["kv_cache"].view(torch.int16))


def test_epilogue_index_rules():
    w = wl.EpiWorkload("bad", T=40, num_kv_heads=1, max_pos=256, num_pages=8, seed=4100)
    inp = wl.make_epi_inputs(w)
    inp["slots"][3] = -1
    inp["slots"][7] = w.num_pages * 16 + 2
    inp["positions"][11] = w.max_pos + 1
    g, st, out_ref, cache_ref, err, parent = run_both(inp, 1, cache_parent_pages=2 * w.num_pages)
    assert err == oracle.ERR_SLOT | oracle.ERR_POSITION
    assert st == qf.STATUS_BAD_SLOT | qf.STATUS_BAD_POSITION
    assert int(parent[w.num_pages:].view(torch.int16).abs().sum()) == 0, "insert past the cache"
    got = wl.bits(g["qkv"].cpu())
    assert np.array_equal(got[11], wl.bits(inp["qkv"])[11])    # bad position: row untouched
    check(inp, 1, g, out_ref, cache_ref)


def test_epilogue_zero_tokens():
    w = wl.EPI_WORKLOADS["epi_t17_nkv1"]
    inp = wl.make_epi_inputs(w)
    g = {k: v.to("cuda:0") for k, v in inp.items()}
    before = g["kv_cache"].clone()
    qf.qknorm_rope_kv_insert(g["qkv"][:0], g["positions"][:0], g["slots"][:0], g["cos_sin"],
                             g["kv_cache"])
    torch.cuda.synchronize()
    assert torch.equal(before, g["kv_cache"])


def test_epilogue_repeat_runs_bitwise_equal():
    w = wl.EPI_WORKLOADS["epi_t1000_nkv8"]
    inp = wl.make_epi_inputs(w)
    outs = []
    for _ in range(2):
        g = {k: v.to("cuda:0") for k, v in inp.items()}
        qf.qknorm_rope_kv_insert(g["qkv"], g["positions"], g["slots"], g["cos_sin"], g["kv_cache"])
        torch.cuda.synchronize()
        outs.append((g["qkv"].clone(), g["kv_cache"].clone()))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))


def test_front_and_epilogue_agree_on_the_same_rows():
    """The fused front's q/k columns equal the standalone epilogue applied to
    the front's own v-and-gate-free projection: run the front on integer
    inputs (exact projection), rebuild the projection from the oracle's exact
    sums, apply the standalone kernel, and compare bit for bit."""
    w = wl.WORKLOADS["m8_nkv8_n9216"]
    inp = wl.make_inputs(w, integer_valued=True)
    g = {k: v.to("cuda:0") for k, v in inp.items()}
    out = qf.qkv_front(g["x"], g["W"], g["positions"], g["slots"], g["cos_sin"], g["kv_cache"])
    p = (inp["x"].double() @ inp["W"].double().T).float().to(torch.bfloat16).to("cuda:0")
    cache2 = inp["kv_cache"].to("cuda:0")
    qf.qknorm_rope_kv_insert(p, g["positions"], g["slots"], g["cos_sin"], cache2)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), p.view(torch.int16))
    assert torch.equal(g["kv_cache"].view(torch.int16), cache2.view(torch.int16))
