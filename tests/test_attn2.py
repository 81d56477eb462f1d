"""attn2 (verify-step paged attention + o-norm + sigmoid gate) through the C
ABI against the oracle: every workload, every cluster split, windows, bad
requests, and the decode layer's order — the front fills the cache and its
q / gate columns, attn2 reads them."""
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


def _dev(inp):
    return {k: v.to("cuda:0") for k, v in inp.items()}


def _oracle(inp, w, window=None, out_bits=None):
    return oracle.attn2(wl.bits(inp["qkv"]), wl.bits(inp["kv_cache"]), inp["block_table"].numpy(),
                        inp["context_lens"].numpy(), w.num_kv_heads,
                        w.window if window is None else window, out_bits=out_bits)


@pytest.mark.parametrize("name", list(wl.ATTN_WORKLOADS))
def test_attn2_workloads_match_oracle(name):
    w = wl.ATTN_WORKLOADS[name]
    inp = wl.make_attn_inputs(w)
    g = _dev(inp)
    out = qf.attn2(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], window=w.window)
    torch.cuda.synchronize()
    assert qf.status() == 0
    ref, err = _oracle(inp, w)
    assert err == 0
    assert_values(wl.bits(out.cpu()), ref, what=f"attn2 {name}")


def test_attn2_default_splits():
    """The split rule on this device: doubled while the grid fits one CTA per
    SM and each split keeps two or more of the pages a row can see, up to 8."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert sms >= 128   # the cases below assume a full GB300
    assert qf.attn2_splits(1, 8, 2048) == 8        # one 32K request: 8 x 8 CTAs
    assert qf.attn2_splits(8, 8, 256) == 2         # 8 requests of 4K: 64 x 2 CTAs
    assert qf.attn2_splits(2, 8, 64, 128) == 4     # window 128: at most 10 pages a row sees
    assert qf.attn2_splits(1, 1, 3) == 1           # too few pages to split
    assert qf.attn2_splits(1, 1, 8) == 4           # two pages per split
    assert qf.attn2_splits(1, 1, 7) == 2
    assert qf.attn2_splits(1, 8, 0) == 0           # bad input


@pytest.mark.parametrize("splits", [1, 2, 4, 8, 16])
def test_attn2_every_split(splits):
    w = wl.ATTN_WORKLOADS["attn_r2_window_nkv8"]
    inp = wl.make_attn_inputs(w)
    g = _dev(inp)
    outs = []
    for _ in range(2):
        outs.append(qf.attn2(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"],
                             window=w.window, splits=splits).clone())
    torch.cuda.synchronize()
    assert qf.status() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref, _ = _oracle(inp, w)
    assert_values(wl.bits(outs[0].cpu()), ref, what=f"attn2 splits={splits}")


@pytest.mark.parametrize("window", [1, 7, 16, 33])
def test_attn2_windows(window):
    w = wl.AttnWorkload(f"w{window}", R=3, num_kv_heads=2, context=(8, 45, 130), num_pages=64,
                        seed=6000 + window, window=window)
    inp = wl.make_attn_inputs(w)
    g = _dev(inp)
    out = qf.attn2(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], window=window)
    torch.cuda.synchronize()
    ref, _ = _oracle(inp, w)
    assert_values(wl.bits(out.cpu()), ref, what=f"attn2 window={window}")


@pytest.mark.parametrize("L", [8, 9, 15, 16, 17, 31, 33, 255, 257])
def test_attn2_lengths_around_page_edges(L):
    w = wl.AttnWorkload(f"l{L}", R=1, num_kv_heads=1, context=(L,), num_pages=32, seed=6100 + L)
    inp = wl.make_attn_inputs(w)
    g = _dev(inp)
    out = qf.attn2(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"])
    torch.cuda.synchronize()
    ref, _ = _oracle(inp, w)
    assert_values(wl.bits(out.cpu()), ref, what=f"attn2 L={L}")


def test_attn2_bad_requests_skipped_and_flagged():
    w = wl.AttnWorkload("bad", R=3, num_kv_heads=1, context=(40, 40, 40), num_pages=16, seed=6200)
    inp = wl.make_attn_inputs(w)
    inp["context_lens"][0] = 5                      # fewer than 8 tokens
    inp["block_table"][1, 1] = 999                  # a page outside the cache
    g = _dev(inp)
    out = torch.full((24, 512), 7.0, dtype=torch.bfloat16, device="cuda:0")
    qf.attn2(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], out=out)
    torch.cuda.synchronize()
    assert qf.status() == qf.STATUS_BAD_REQUEST
    got = wl.bits(out.cpu())
    assert np.all(got[:16] == wl.bits(torch.tensor([7.0]).to(torch.bfloat16))[0])
    ref, err = _oracle(inp, w)
    assert err == oracle.ERR_ATTN_REQUEST
    assert_values(got[16:], ref[16:], what="the good request")


def test_decode_layer_front_then_attn2():
    """The order of a decode layer: the front writes q / gate and inserts K / V
    for the 8 verify tokens, then attn2 reads them (PDL-linked on one stream),
    against the oracle front followed by the oracle attn2."""
    nkv, L = 2, 300
    w = wl.Workload("layer", M=8, num_kv_heads=nkv, max_pos=4096, num_pages=64, seed=6300)
    inp = wl.make_inputs(w)
    table = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(1))[:(L + 15) // 16]
    table = table.to(torch.int32)[None, :]
    slots = torch.tensor([int(table[0, j // 16]) * 16 + j % 16 for j in range(L - 8, L)])
    inp["slots"] = slots
    inp["positions"] = torch.arange(L - 8, L)
    lens = torch.tensor([L], dtype=torch.int32)
    g = _dev(inp)
    gt, gl = table.to("cuda:0"), lens.to("cuda:0")
    qkv = qf.qkv_front(g["x"], g["W"], g["positions"], g["slots"], g["cos_sin"], g["kv_cache"])
    o = qf.attn2(qkv, g["kv_cache"], gt, gl)
    torch.cuda.synchronize()
    assert qf.status() == 0
    cache_ref = wl.bits(inp["kv_cache"]).copy()
    out_ref, err = oracle.qkv_front(wl.bits(inp["x"]), wl.bits(inp["W"]), inp["positions"].numpy(),
                                    slots.numpy(), inp["cos_sin"].numpy(), cache_ref, nkv)
    assert err == 0
    # attn2 against the oracle on the GPU's own front output and cache (isolates attn2)
    o_ref, err = oracle.attn2(wl.bits(qkv.cpu()), wl.bits(g["kv_cache"].cpu()), table.numpy(),
                              lens.numpy(), nkv)
    assert err == 0
    assert_values(wl.bits(o.cpu()), o_ref, what="attn2 after the front")
    # and the whole layer against the all-oracle chain
    o_chain, _ = oracle.attn2(out_ref, cache_ref, table.numpy(), lens.numpy(), nkv)
    assert_values(wl.bits(o.cpu()), o_chain, what="front + attn2 vs the oracle chain")


# ---- the split-KV engine: partials in a caller's workspace, a second grid merges ----

def _workspace(R, nkv, splits):
    """A workspace of the size asked for, filled with NaN bytes: the engine
    needs no initial contents."""
    n = qf.attn2_split_kv_workspace_bytes(R, nkv, splits)
    assert n > 0
    return torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda:0")


@pytest.mark.parametrize("name", list(wl.ATTN_WORKLOADS))
def test_attn2_split_kv_workloads_match_oracle(name):
    w = wl.ATTN_WORKLOADS[name]
    inp = wl.make_attn_inputs(w)
    g = _dev(inp)
    S = qf.attn2_split_kv_splits(w.R, w.num_kv_heads, w.max_blocks(), w.window)
    assert S >= 1
    ws = _workspace(w.R, w.num_kv_heads, S)
    out = qf.attn2_split_kv(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], ws,
                            window=w.window)
    torch.cuda.synchronize()
    assert qf.status() == 0
    ref, err = _oracle(inp, w)
    assert err == 0
    assert_values(wl.bits(out.cpu()), ref, what=f"attn2 split-KV {name} S={S}")


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8, 19, 40])
@pytest.mark.parametrize("name", ["attn_r3_mixed_nkv2", "attn_r2_window_nkv8"])
def test_attn2_split_kv_every_split(name, splits):
    """Any split, including more CTAs than pages (empty partials), matches the
    oracle and repeats bitwise."""
    w = wl.ATTN_WORKLOADS[name]
    inp = wl.make_attn_inputs(w)
    g = _dev(inp)
    ws = _workspace(w.R, w.num_kv_heads, splits)
    outs = []
    for _ in range(2):
        outs.append(qf.attn2_split_kv(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"],
                                      ws, window=w.window, splits=splits).clone())
    torch.cuda.synchronize()
    assert qf.status() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref, _ = _oracle(inp, w)
    assert_values(wl.bits(outs[0].cpu()), ref, what=f"attn2 split-KV {name} S={splits}")


def test_attn2_split_kv_agrees_with_cluster_engine():
    """Both engines at the same split: the same rows to the tolerance (their
    merge orders differ only in the split partials' summation)."""
    w = wl.ATTN_WORKLOADS["attn_r8_l4k_nkv8"]
    inp = wl.make_attn_inputs(w)
    g = _dev(inp)
    a = qf.attn2(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], splits=2)
    ws = _workspace(w.R, w.num_kv_heads, 2)
    b = qf.attn2_split_kv(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], ws, splits=2)
    torch.cuda.synchronize()
    assert qf.status() == 0
    ref, _ = _oracle(inp, w)
    assert_values(wl.bits(a.cpu()), ref, what="cluster engine")
    assert_values(wl.bits(b.cpu()), ref, what="split-KV engine")


def test_attn2_split_kv_bad_requests_skipped_and_flagged():
    w = wl.AttnWorkload("bad", R=3, num_kv_heads=1, context=(40, 40, 40), num_pages=16, seed=6200)
    inp = wl.make_attn_inputs(w)
    inp["context_lens"][0] = 5
    inp["block_table"][1, 1] = 999
    g = _dev(inp)
    out = torch.full((24, 512), 7.0, dtype=torch.bfloat16, device="cuda:0")
    ws = _workspace(w.R, 1, 3)
    qf.attn2_split_kv(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], ws, out=out,
                      splits=3)
    torch.cuda.synchronize()
    assert qf.status() == qf.STATUS_BAD_REQUEST
    got = wl.bits(out.cpu())
    assert np.all(got[:16] == wl.bits(torch.tensor([7.0]).to(torch.bfloat16))[0])
    ref, _ = _oracle(inp, w)
    assert_values(got[16:], ref[16:], what="the good request")


def test_attn2_split_kv_short_workspace_refused():
    w = wl.ATTN_WORKLOADS["attn_r1_l8_nkv1"]
    g = _dev(wl.make_attn_inputs(w))
    ws = _workspace(w.R, 1, 4)
    with pytest.raises(qf.QkvFrontError):
        qf.attn2_split_kv(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], ws[:-16],
                          splits=4)


def test_attn2_two_ctas_per_sm_shape():
    """A direct launch with more (request, KV head) pairs than SMs runs the
    two-CTA-per-SM shape (2 compute groups, a 4-block ring): 160 requests of
    mixed lengths with a window, one request too short and one with a table
    entry outside the cache, through both entry points, against the oracle
    and bitwise on a repeat."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    R = sms + 8
    rng = np.random.default_rng(6600)
    ctx = tuple(int(x) for x in rng.integers(8, 200, size=R))
    w = wl.AttnWorkload("two_per_sm", R=R, num_kv_heads=1, context=ctx,
                        num_pages=sum((c + 15) // 16 for c in ctx) + 8, seed=6601, window=40)
    inp = wl.make_attn_inputs(w)
    inp["context_lens"][3] = 5
    inp["block_table"][7, (int(inp["context_lens"][7]) - 1) // 16] = w.num_pages + 3   # its last page: visible
    g = _dev(inp)
    fill = torch.full((8 * R, 512), 7.0, dtype=torch.bfloat16, device="cuda:0")
    outs = []
    for _ in range(2):
        outs.append(qf.attn2(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], out=fill.clone(),
                             window=w.window, splits=1))
    ws = torch.zeros(qf.attn2_split_kv_workspace_bytes(R, 1, 1), dtype=torch.uint8, device="cuda:0")
    outs.append(qf.attn2_split_kv(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], ws,
                                  out=fill.clone(), window=w.window, splits=1))
    torch.cuda.synchronize()
    assert qf.status() == qf.STATUS_BAD_REQUEST
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))
    got = wl.bits(outs[0].cpu())
    seven = wl.bits(torch.tensor([7.0]).to(torch.bfloat16))[0]
    assert np.all(got[24:32] == seven) and np.all(got[56:64] == seven)   # requests 3 and 7 skipped
    ref, _ = _oracle(inp, w)
    keep = np.ones(8 * R, dtype=bool)
    keep[24:32] = False
    keep[56:64] = False
    assert_values(got[keep], ref[keep], what="attn2, two CTAs per SM")


def test_attn2_most_kv_heads():
    """64 KV heads (512 q heads, out rows of 32768 columns): the cluster engine
    at its own split and at two, the direct launch (192 pairs: the
    two-CTA-per-SM shape) and the split-KV engine, against the oracle."""
    w = wl.AttnWorkload("r3_nkv64", R=3, num_kv_heads=64, context=(8, 77, 300), num_pages=64,
                        seed=6700)
    inp = wl.make_attn_inputs(w)
    g = _dev(inp)
    outs = {
        "attn2": qf.attn2(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"]),
        "attn2 splits=2": qf.attn2(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], splits=2),
        "attn2 splits=1": qf.attn2(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], splits=1),
    }
    S = qf.attn2_split_kv_splits(w.R, w.num_kv_heads, w.max_blocks(), w.window)
    ws = _workspace(w.R, w.num_kv_heads, S)
    outs[f"split-KV S={S}"] = qf.attn2_split_kv(g["qkv"], g["kv_cache"], g["block_table"],
                                                g["context_lens"], ws)
    torch.cuda.synchronize()
    assert qf.status() == 0
    ref, err = _oracle(inp, w)
    assert err == 0
    for what, out in outs.items():
        assert out.shape == (24, 32768)
        assert_values(wl.bits(out.cpu()), ref, what=what)
