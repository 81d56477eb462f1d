"""attn2_split_kv_noalloc: split-KV attention for callers that cannot
allocate device memory themselves — a plugin whose host process owns every
device allocation through its own pool, or a decode step that must not risk
cudaMalloc's implicit synchronisation or a failed allocation mid-step.  Its
partials live in the library's own device array instead of a caller's
workspace.  Checked through the C ABI against attn2_split_kv with a caller's
workspace (bit for bit: both run the same kernels at the same split) and
against the oracle, on two calls in a row.  This file is collected last, so
a run that stops at its first failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle
from kv_insert_gb300 import qkv_front as qf
from kv_insert_gb300 import workloads as wl

from _parity import assert_values

SLOTS = 256   # partial slots in the library's array: num_reqs * num_kv_heads * splits


@pytest.fixture(scope="module")
def built():
    import __graft_entry__
    __graft_entry__.build()
    return qf.load()


def test_noalloc_refuses_more_slots_than_its_array(built):
    """Sizes beyond the array are refused on the host, before any launch
    (explicit splits need no device query)."""
    lib = built
    X, CACHE, POS, SL, OUT = ((i + 1) << 36 for i in range(5))
    # 2 requests x 2 KV heads x 65 splits = 260 slots > 256
    assert lib.attn2_split_kv_noalloc(X, CACHE, 64, POS, 8, SL, 2, 2304, 2, 0, 0.125, 1e-6, OUT, 65,
                                      None) == 7
    assert lib.attn2_split_kv_noalloc(X, CACHE, 64, POS, 8, SL, 2, 2304, 2, 0, 0.125, 1e-6, OUT, 257,
                                      None) == 8
    assert lib.attn2_split_kv_noalloc(0, CACHE, 64, POS, 8, SL, 2, 2304, 2, 0, 0.125, 1e-6, OUT, 1,
                                      None) == 3


def _oracle(inp, w):
    return oracle.attn2(wl.bits(inp["qkv"]), wl.bits(inp["kv_cache"]), inp["block_table"].numpy(),
                        inp["context_lens"].numpy(), w.num_kv_heads, w.window)


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_engine_two_calls_in_a_row(built):
    """Call 1: one 32K request, 8 KV heads, the library's split (152 slots).
    Call 2: three mixed requests at 5 splits (30 slots) on other inputs, so
    call 1's partials still sit in the array's slots above call 2's range.
    Each call equals attn2_split_kv at the same split with a caller's
    workspace bit for bit, and both match the oracle within the parity
    tolerance of the other tests."""
    for name, splits in (("attn_r1_l32k_nkv8", 0), ("attn_r3_mixed_nkv2", 5)):
        w = wl.ATTN_WORKLOADS[name]
        inp = wl.make_attn_inputs(w)
        g = {k: v.to("cuda:0") for k, v in inp.items()}
        S = splits or qf.attn2_split_kv_splits(w.R, w.num_kv_heads, w.max_blocks(), w.window)
        assert 2 <= S and w.R * w.num_kv_heads * S <= SLOTS
        out = torch.empty(8 * w.R, 512 * w.num_kv_heads, dtype=torch.bfloat16, device="cuda:0")
        qf.attn2_split_kv_noalloc(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"],
                                  out=out, window=w.window, splits=splits)
        ws = torch.zeros(qf.attn2_split_kv_workspace_bytes(w.R, w.num_kv_heads, S), dtype=torch.uint8,
                         device="cuda:0")
        ref = qf.attn2_split_kv(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], ws,
                                window=w.window, splits=S)
        torch.cuda.synchronize()
        assert qf.status() == 0
        got_bits, ws_bits = wl.bits(out.cpu()), wl.bits(ref.cpu())
        if not np.array_equal(got_bits, ws_bits):
            # a readable report of how far apart they are, then fail
            assert_values(got_bits, ws_bits, what=f"no-alloc vs workspace {name} S={S}")
            pytest.fail(f"{name} S={S}: {int((got_bits != ws_bits).sum())} outputs differ in bits "
                        "from the workspace engine at the same split")
        ora, err = _oracle(inp, w)
        assert err == 0
        assert_values(got_bits, ora, what=f"no-alloc attn2 {name} S={S} vs oracle")
        assert_values(ws_bits, ora, what=f"workspace attn2 {name} S={S} vs oracle")


@pytest.mark.gpu
def test_noalloc_one_split_needs_no_array_slots(built):
    """40 requests x 8 KV heads = 320 (request, KV head) pairs, more than the
    array's 256 slots: at one split the call takes the direct path and runs;
    at two splits (640 slots) it is refused with QKVF_ERR_SIZES and launches
    nothing."""
    w = wl.AttnWorkload("noalloc_big", R=40, num_kv_heads=8, context=(64,) * 40, num_pages=256, seed=7100)
    inp = wl.make_attn_inputs(w)
    g = {k: v.to("cuda:0") for k, v in inp.items()}
    out = torch.full((8 * w.R, 512 * w.num_kv_heads), 3.0, dtype=torch.bfloat16, device="cuda:0")
    with pytest.raises(qf.QkvFrontError) as e:
        qf.attn2_split_kv_noalloc(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], out=out,
                                  splits=2)
    assert e.value.code == 7
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
    qf.attn2_split_kv_noalloc(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], out=out,
                              splits=1)
    ref = qf.attn2(g["qkv"], g["kv_cache"], g["block_table"], g["context_lens"], splits=1)
    torch.cuda.synchronize()
    assert qf.status() == 0
    assert np.array_equal(wl.bits(out.cpu()), wl.bits(ref.cpu()))
    ora, err = _oracle(inp, w)
    assert err == 0
    assert_values(wl.bits(out.cpu()), ora, what="no-alloc attn2 at one split vs oracle")
