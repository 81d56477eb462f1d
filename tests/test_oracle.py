"""Pins of the CPU oracle to facts other than itself (no GPU).

Each test ties one oracle step to a property fixed by the pages or by the
mathematics: hand-derived golden values, a library routine on a special
case, exact integer arithmetic, closed forms, invariants, brute-force scans.
A plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, eps in the wrong place, a sum for a mean, neox pairing,
a k/v swap) fails at least one of them; the comment on each test says which.
"""
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle
from kv_insert_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_bits(values):
    return np.asarray(values, dtype=np.float32).view(np.uint32)


def bits_to_f32(u32):
    return np.asarray(u32, dtype=np.uint32).view(np.float32)


# ---- BF16 rounding -------------------------------------------------------

def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append((int(parts[0], 16), int(parts[1], 16), " ".join(parts[2:])))
    return rows


def test_bf16_rne_golden(oracle_lib):
    """Hand-derived ties-to-even cases (ties, carries, overflow, subnormals, NaN)."""
    for f_bits, want, note in _golden_rows("bf16_rne.txt"):
        f = struct.unpack("<f", struct.pack("<I", f_bits))[0]
        got = int(oracle.f32_to_bf16_bits(np.float32(f)))
        if (want & 0x7F80) == 0x7F80 and (want & 0x7F) != 0:
            assert (got & 0x7F80) == 0x7F80 and (got & 0x7F) != 0, note
        else:
            assert got == want, f"{note}: {f_bits:#010x} -> {got:#06x}, want {want:#06x}"


def test_bf16_rne_matches_torch(oracle_lib):
    """torch's float->bfloat16 cast is round-to-nearest-even: same bits on
    random patterns of every class (normal, subnormal, huge, ties)."""
    rng = np.random.default_rng(7)
    pats = rng.integers(0, 2**32, size=6000, dtype=np.uint64).astype(np.uint32)
    ties = (pats & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    small = pats & np.uint32(0x807FFFFF)             # subnormals
    vals = bits_to_f32(np.concatenate([pats, ties, small]))
    vals = vals[np.isfinite(vals)]
    got = oracle.f32_to_bf16_bits(vals)
    want = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    nan = bits_to_f32(np.array([0x7FC00000, 0xFFC00001, 0x7F800001], dtype=np.uint32))
    assert np.all(np.isnan(oracle.bf16_bits_to_f32(oracle.f32_to_bf16_bits(nan))))


def test_bf16_widening_exact(oracle_lib):
    """bf16 -> fp32 is the bit pattern shifted up (every bf16 value is an fp32 value)."""
    allbits = np.arange(0, 65536, 97, dtype=np.uint16)
    got = oracle.bf16_bits_to_f32(allbits)
    want = bits_to_f32(allbits.astype(np.uint32) << 16)
    # NaN payloads are quieted by the Python float round trip of the wrapper,
    # so NaN patterns are only checked to stay NaN
    nan = np.isnan(want)
    assert np.array_equal(got.view(np.uint32)[~nan], want.view(np.uint32)[~nan])
    assert np.all(np.isnan(got[nan]))


# ---- projection -------------------------------------------------------------

@pytest.mark.parametrize("K", [64, 8192])
def test_project_integer_exact(oracle_lib, K):
    """With integer x, W in [-4, 4] every partial sum is an integer below 2^24,
    so FP32 accumulation is exact in any order: acc must equal the int64
    matmul x @ W^T.  A transposed operand or a dropped term fails."""
    rng = np.random.default_rng(K)
    M, N = 3, 72
    xi = rng.integers(-4, 5, size=(M, K))
    wi = rng.integers(-4, 5, size=(N, K))
    xb = wl.bits(torch.from_numpy(xi.astype(np.float32)).to(torch.bfloat16))
    wb = wl.bits(torch.from_numpy(wi.astype(np.float32)).to(torch.bfloat16))
    acc = oracle.project_f32(xb, wb)
    exact = xi @ wi.T
    assert np.array_equal(acc.astype(np.int64), exact)
    assert np.array_equal(acc, exact.astype(np.float32))


def test_project_float_error_bound(oracle_lib):
    """Random normal inputs: |acc - exact| <= gamma_K * sum|x||w| with
    gamma_K = K u / (1 - K u), u = 2^-24 (the standard bound for recursive
    summation of rounded products), against a float64 library matmul."""
    rng = np.random.default_rng(3)
    M, N, K = 4, 40, 8192
    x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy((rng.standard_normal((N, K)) / math.sqrt(K)).astype(np.float32)).to(torch.bfloat16)
    acc = oracle.project_f32(wl.bits(x), wl.bits(w))
    xd, wd = x.double().numpy(), w.double().numpy()
    exact = xd @ wd.T
    u = 2.0 ** -24
    gamma = K * u / (1 - K * u)
    bound = gamma * (np.abs(xd) @ np.abs(wd).T)
    assert np.all(np.abs(acc.astype(np.float64) - exact) <= bound)
    # and the rows are not a permutation of one another (catches t/n swaps)
    assert not np.allclose(acc[0], acc[1])


# ---- head layout ---------------------------------------------------------

@pytest.mark.parametrize("nkv", [1, 2, 8, 16])
def test_head_kind_matches_split_qkv_views(oracle_lib, nkv):
    """cute_ops page, split_qkv: the q view is columns [0, q_width), the gate
    view [q_width + 2 kv_width, N) with q_width = 8 * nkv * 64; k precedes v."""
    N = wl.columns_for(nkv)
    q_width, kv_width = 8 * nkv * 64, nkv * 64
    assert N == 2 * q_width + 2 * kv_width
    for h in range(N // 64):
        col = h * 64
        kind = oracle.head_kind(h, nkv)
        if col < q_width:
            assert kind == oracle.HEAD_Q
        elif col >= q_width + 2 * kv_width:
            assert kind == oracle.HEAD_GATE
        elif col < q_width + kv_width:
            assert kind == oracle.HEAD_K
        else:
            assert kind == oracle.HEAD_V


# ---- RMS norm --------------------------------------------------------------

@pytest.mark.parametrize("c", [2.0 ** -10, 1e-3, 0.37, 3.0, 100.0, -5.5])
def test_norm_constant_closed_form(oracle_lib, c):
    """A constant head c normalises to c / sqrt(c^2 + eps) (mean of 64 equal
    squares is c^2).  eps outside the root, or a sum for the mean, fails
    (visible at small c where eps matters)."""
    p = np.full(64, c, dtype=np.float32)
    u = oracle.rms_norm_head(p)
    cf = float(np.float32(c))
    want = cf / math.sqrt(cf * cf + 1e-6)
    assert np.all(np.abs(u.astype(np.float64) - want) <= 4 * 2.0 ** -24 * abs(want))


def test_norm_rms_invariant(oracle_lib):
    """RMS of the normed head = sqrt(ms / (ms + eps)), i.e. 1 within eps."""
    rng = np.random.default_rng(11)
    for scale in (1e-2, 1.0, 37.0):
        p = (rng.standard_normal(64) * scale).astype(np.float32)
        u = oracle.rms_norm_head(p).astype(np.float64)
        ms = np.mean(p.astype(np.float64) ** 2)
        rms = math.sqrt(np.mean(u ** 2))
        assert abs(rms - math.sqrt(ms / (ms + 1e-6))) <= 1e-6
        assert abs(rms - 1.0) <= 1e-6 / ms + 1e-6


def test_norm_scale_invariance_and_direction(oracle_lib):
    """norm(2^k p) / norm(p) = sqrt((ms + eps) / (ms + eps 4^-k)) (the eps term
    is the only scale dependence), and u is a positive multiple of p."""
    rng = np.random.default_rng(12)
    p = rng.standard_normal(64).astype(np.float32)
    base = oracle.rms_norm_head(p).astype(np.float64)
    ms = float(np.mean(p.astype(np.float64) ** 2))
    for k in (-3, -1, 2, 5):
        scaled = oracle.rms_norm_head((p * np.float32(2.0 ** k)).astype(np.float32))
        want = math.sqrt((ms + 1e-6) / (ms + 1e-6 * 4.0 ** -k))
        assert np.allclose(scaled / base, want, rtol=2e-6, atol=0)
    ratio = base.astype(np.float64) / p.astype(np.float64)
    assert np.all(ratio > 0) and np.ptp(ratio) <= 1e-6 * ratio.mean()


# ---- interleaved RoPE -----------------------------------------------------

def _row(cos, sin):
    return np.concatenate([np.asarray(cos, np.float32), np.asarray(sin, np.float32)])


def test_rope_identity_row(oracle_lib):
    """A row of cos 1 / sin 0 (position 0 of any base) leaves the head unchanged."""
    u = np.random.default_rng(1).standard_normal(64).astype(np.float32)
    y = oracle.rope_head(u, _row(np.ones(32), np.zeros(32)))
    assert np.array_equal(y.view(np.uint32), u.view(np.uint32))


def test_rope_quarter_turn_pins_pairs_and_sign(oracle_lib):
    """cos 0 / sin 1 turns each pair (u_2i, u_2i+1) to (-u_2i+1, u_2i) exactly.
    A neox pairing (i, i + 32) or the opposite sign gives other values."""
    u = np.random.default_rng(2).standard_normal(64).astype(np.float32)
    y = oracle.rope_head(u, _row(np.zeros(32), np.ones(32)))
    want = np.empty(64, np.float32)
    want[0::2] = -u[1::2]
    want[1::2] = u[0::2]
    assert np.array_equal(y, want)


def test_rope_half_turn_negates(oracle_lib):
    u = np.random.default_rng(3).standard_normal(64).astype(np.float32)
    y = oracle.rope_head(u, _row(-np.ones(32), np.zeros(32)))
    assert np.array_equal(y, -u)


def test_rope_per_pair_angles_geometric(oracle_lib):
    """Pair i turns by its own angle theta_i (read from column i and 32 + i):
    its length is kept and atan2 grows by theta_i (checked in float64)."""
    rng = np.random.default_rng(4)
    u = rng.standard_normal(64).astype(np.float32)
    theta = rng.uniform(-math.pi, math.pi, 32)
    y = oracle.rope_head(u, _row(np.cos(theta), np.sin(theta))).astype(np.float64)
    a, b = u[0::2].astype(np.float64), u[1::2].astype(np.float64)
    y0, y1 = y[0::2], y[1::2]
    assert np.allclose(np.hypot(y0, y1), np.hypot(a, b), rtol=1e-6, atol=1e-7)
    turn = np.angle(np.exp(1j * (np.arctan2(y1, y0) - np.arctan2(b, a) - theta)))
    assert np.all(np.abs(turn) < 1e-5)


def test_rope_table_closed_form():
    """The workload table is cos/sin(pos * 10000^(-2i/64)) in columns i | 32 + i."""
    tab = wl.rope_table(4096).numpy().astype(np.float64)
    for pos in (0, 1, 17, 4095):
        for i in (0, 5, 31):
            ang = pos * 10000.0 ** (-2.0 * i / 64)
            assert abs(tab[pos, i] - math.cos(ang)) <= 1e-7
            assert abs(tab[pos, 32 + i] - math.sin(ang)) <= 1e-7
    assert np.all(tab[0, :32] == 1.0) and np.all(tab[0, 32:] == 0.0)


# ---- paged K/V insert ----------------------------------------------------

def test_kv_insert_bruteforce_placement(oracle_lib):
    """Scan the whole cache after each insert: exactly the 2 x nkv x 64 elements
    of (page = slot / 16, offset = slot % 16) change; the K half holds the k
    head columns of the row and the V half its v head columns."""
    nkv, pages = 2, 4
    N = wl.columns_for(nkv)
    rng = np.random.default_rng(5)
    row = rng.integers(0, 65536, size=N, dtype=np.uint64).astype(np.uint16)
    q_width, kv_width = 8 * nkv * 64, nkv * 64
    for slot in range(pages * 16):
        cache = rng.integers(0, 65536, size=(pages, nkv, 16, 128), dtype=np.uint64).astype(np.uint16)
        before = cache.copy()
        oracle.kv_insert_token(row, slot, cache, nkv)
        changed = np.argwhere(cache != before)
        for pg, g, off, _ in changed:
            assert pg * 16 + off == slot
        page, off = divmod(slot, 16)
        for g in range(nkv):
            assert np.array_equal(cache[page, g, off, :64], row[q_width + g * 64: q_width + g * 64 + 64])
            assert np.array_equal(cache[page, g, off, 64:],
                                  row[q_width + kv_width + g * 64: q_width + kv_width + g * 64 + 64])
        mask = np.ones(cache.shape, bool)
        mask[page, :, off, :] = False
        assert np.array_equal(cache[mask], before[mask])


# ---- the whole front ------------------------------------------------------

def _bf(values):
    return wl.bits(torch.tensor(np.asarray(values, np.float32)).to(torch.bfloat16))


def _worked_case():
    nkv = 1
    N = wl.columns_for(nkv)
    w = np.zeros(N, np.float32)
    w[0] = 8.0                                   # head 0 (q): (8, 0, ..., 0)
    w[8 * 64: 9 * 64] = 2.0 ** -10               # head 8 (k): constant 2^-10
    w[9 * 64: 10 * 64] = (np.arange(64) + 1) / 8.0   # head 9 (v)
    for h in range(10, 18):                      # gate heads
        w[h * 64: h * 64 + 64] = -h / 4.0
    x = _bf([[1.0]])
    W = _bf(w[:, None])
    cs = np.zeros((1, 64), np.float32)
    cs[0, :32] = 1.0
    cs[0, 0] = 0.0
    cs[0, 32] = 1.0
    cache = np.full((2, 1, 16, 128), 0x1234, np.uint16)
    return x, W, cs, cache, w


def test_full_worked_example_golden(oracle_lib):
    """tests/golden/head_epilogue.txt, derived by hand: rounding, norm (mean,
    eps inside the root), quarter-turn RoPE on pair 0, pass-through of v and
    gate, and the insert at slot 21 -> page 1, offset 5."""
    x, W, cs, cache, w = _worked_case()
    out, err = oracle.qkv_front(x, W, [0], [21], cs, cache, 1)
    assert err == 0
    want = {}
    for line in open(os.path.join(GOLDEN, "head_epilogue.txt")):
        if line.startswith("head"):
            name, a, b, rest = line.split()
            n, v = rest.split("x", 1)
            want[name] = [int(a, 16), int(b, 16)] + [int(v, 16)] * int(n)
    assert out[0, 0:64].tolist() == want["head0"]
    assert out[0, 8 * 64: 9 * 64].tolist() == want["head8"]
    assert np.array_equal(out[0, 9 * 64: 10 * 64], _bf(w[9 * 64: 10 * 64]))
    assert np.array_equal(out[0, 10 * 64:], _bf(w[10 * 64:]))
    assert np.array_equal(cache[1, 0, 5, :64], out[0, 8 * 64: 9 * 64])
    assert np.array_equal(cache[1, 0, 5, 64:], out[0, 9 * 64: 10 * 64])
    untouched = np.ones(cache.shape, bool)
    untouched[1, 0, 5] = False
    assert np.all(cache[untouched] == 0x1234)


@pytest.mark.parametrize("nkv", [1, 2, 3])
def test_full_which_heads_are_normed(oracle_lib, nkv):
    """Give head h the constant (2h + 3)/16 (never 1.0) and use the identity
    row: a normed head becomes all 1.0 (c^2 >> eps), a passed-through head
    keeps its constant.  The normed set must be exactly the q and k heads
    (columns before q_width + kv_width, split_qkv)."""
    N = wl.columns_for(nkv)
    heads = N // 64
    consts = (2 * np.arange(heads) + 3) / 16.0
    W = _bf(np.repeat(consts, 64)[:, None])
    cs = _row(np.ones(32), np.zeros(32))[None, :]
    cache = np.zeros((1, nkv, 16, 128), np.uint16)
    out, err = oracle.qkv_front(_bf([[1.0]]), W, [0], [3], cs, cache, nkv)
    assert err == 0
    one = int(_bf([1.0])[0])
    q_width, kv_width = 8 * nkv * 64, nkv * 64
    for h in range(heads):
        seg = out[0, h * 64:(h + 1) * 64]
        if h * 64 < q_width + kv_width:
            assert np.all(seg == one), h
        else:
            assert np.all(seg == int(_bf([consts[h]])[0])), h
    for g in range(nkv):
        assert np.all(cache[0, g, 3, :64] == one)
        assert np.all(cache[0, g, 3, 64:] == int(_bf([consts[9 * nkv + g]])[0]))


def test_full_integer_inputs_pass_through_bit_exact(oracle_lib):
    """Integer x, W: v and gate columns of out (and the cache V half) are the
    exact integer sums rounded by torch's RNE cast (a library routine)."""
    w = wl.Workload("tiny", M=3, num_kv_heads=1, max_pos=64, num_pages=4, seed=9)
    inp = wl.make_inputs(w, integer_valued=True)
    cache = wl.bits(inp["kv_cache"]).copy()
    out, err = oracle.qkv_front(wl.bits(inp["x"]), wl.bits(inp["W"]), inp["positions"].numpy(),
                                inp["slots"].numpy(), inp["cos_sin"].numpy(), cache, 1)
    assert err == 0
    exact = inp["x"].double() @ inp["W"].double().T
    want = wl.bits(exact.float().to(torch.bfloat16))
    vg = slice(9 * 64, 18 * 64)
    assert np.array_equal(out[:, vg], want[:, vg])
    for t in range(3):
        page, off = divmod(int(inp["slots"][t]), 16)
        assert np.array_equal(cache[page, 0, off, 64:], want[t, 9 * 64: 10 * 64])


def test_full_slot_and_position_rules(oracle_lib):
    """A negative slot inserts nothing (padding); an out-of-range slot inserts
    nothing and reports ERR_SLOT; an out-of-range position leaves the token's
    q and k heads and the cache untouched and reports ERR_POSITION."""
    x, W, cs, cache, w = _worked_case()
    start = np.full((1, wl.columns_for(1)), 0x7777, np.uint16)
    c0 = cache.copy()
    out, err = oracle.qkv_front(x, W, [0], [-1], cs, cache, 1, out_bits=start)
    assert err == 0 and np.array_equal(cache, c0)
    out, err = oracle.qkv_front(x, W, [0], [32], cs, cache, 1, out_bits=start)
    assert err == oracle.ERR_SLOT and np.array_equal(cache, c0)
    out, err = oracle.qkv_front(x, W, [1], [21], cs, cache, 1, out_bits=start)
    assert err == oracle.ERR_POSITION and np.array_equal(cache, c0)
    assert np.all(out[0, : 9 * 64] == 0x7777)
    assert np.array_equal(out[0, 9 * 64:], _bf(w[9 * 64:]))


def test_full_tiny_bruteforce_float64(oracle_lib):
    """Tiny hidden size: the oracle agrees with a float64 restatement of the
    definition within the BF16 rounding of its last step."""
    rng = np.random.default_rng(21)
    nkv, M, K = 1, 3, 16
    N = wl.columns_for(nkv)
    x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy((rng.standard_normal((N, K)) / 4).astype(np.float32)).to(torch.bfloat16)
    pos = np.array([0, 5, 9])
    cs = wl.rope_table(10).numpy()
    cache = np.zeros((2, nkv, 16, 128), np.uint16)
    out, err = oracle.qkv_front(wl.bits(x), wl.bits(W), pos, [0, 17, 31], cs, cache, nkv)
    assert err == 0
    p = (x.double() @ W.double().T).float().to(torch.bfloat16).double().numpy()
    got = wl.from_bits(out).double().numpy()
    for t in range(M):
        for h in range(N // 64):
            seg = p[t, h * 64:(h + 1) * 64]
            if h < 9 * nkv:
                u = seg / math.sqrt(np.mean(seg ** 2) + 1e-6)
                c, s = cs[pos[t], :32].astype(np.float64), cs[pos[t], 32:].astype(np.float64)
                y = np.empty(64)
                y[0::2] = u[0::2] * c - u[1::2] * s
                y[1::2] = u[1::2] * c + u[0::2] * s
                seg = y
            g = got[t, h * 64:(h + 1) * 64]
            assert np.all(np.abs(g - seg) <= 2.0 ** -8 * np.abs(seg) + 1e-6), (t, h)


def test_full_refuses_bad_shape(oracle_lib):
    cache = np.zeros((1, 1, 16, 128), np.uint16)
    x = np.zeros((1, 4), np.uint16)
    W = np.zeros((1000, 4), np.uint16)
    _, err = oracle.qkv_front(x, W, [0], [0], np.zeros((1, 64), np.float32), cache, 1)
    assert err == oracle.ERR_SHAPE


# ---- the unfused epilogue ----------------------------------------------------

def test_unfused_epilogue_composes_to_the_front(oracle_lib):
    """qkv_front page, module docstring: the front writes what the projection
    GEMM followed by fused_muse_spark_qknorm_rope_kv_insert writes.  With the
    same summation order both sides are bitwise equal: out and cache."""
    w = wl.Workload("compose", M=5, num_kv_heads=2, max_pos=512, num_pages=8, seed=31)
    inp = wl.make_inputs(w)
    xb, Wb = wl.bits(inp["x"]), wl.bits(inp["W"])
    pos, sl, cs = inp["positions"].numpy(), inp["slots"].numpy(), inp["cos_sin"].numpy()
    cache_a = wl.bits(inp["kv_cache"]).copy()
    out_a, err_a = oracle.qkv_front(xb, Wb, pos, sl, cs, cache_a, 2)
    p = oracle.f32_to_bf16_bits(oracle.project_f32(xb, Wb))
    cache_b = wl.bits(inp["kv_cache"]).copy()
    out_b, err_b = oracle.qknorm_rope_kv_insert(p, pos, sl, cs, cache_b, 2)
    assert err_a == err_b == 0
    assert np.array_equal(out_a, out_b)
    assert np.array_equal(cache_a, cache_b)


def test_unfused_epilogue_leaves_v_and_gate(oracle_lib):
    """v and gate heads of the projection output are not touched; q and k
    heads are (the identity row makes them normed copies: RMS 1)."""
    rng = np.random.default_rng(8)
    nkv, T = 1, 3
    N = wl.columns_for(nkv)
    qkv = _bf(rng.standard_normal((T, N)) * 3).reshape(T, N)
    cs = _row(np.ones(32), np.zeros(32))[None, :]
    cache = np.zeros((1, nkv, 16, 128), np.uint16)
    out, err = oracle.qknorm_rope_kv_insert(qkv, [0, 0, 0], [-1, -1, -1], cs, cache, nkv)
    assert err == 0
    assert np.array_equal(out[:, 9 * 64:], qkv[:, 9 * 64:])
    assert not np.array_equal(out[:, :9 * 64], qkv[:, :9 * 64])
    vals = wl.from_bits(out[:, :9 * 64]).double().numpy().reshape(T, 9, 64)
    rms = np.sqrt(np.mean(vals ** 2, axis=2))
    assert np.all(np.abs(rms - 1.0) < 1e-2)
    assert not cache.any()


def test_unfused_epilogue_index_rules(oracle_lib):
    nkv, T = 1, 4
    N = wl.columns_for(nkv)
    rng = np.random.default_rng(9)
    qkv = _bf(rng.standard_normal((T, N))).reshape(T, N)
    cs = wl.rope_table(8).numpy()
    cache = np.zeros((2, nkv, 16, 128), np.uint16)
    out, err = oracle.qknorm_rope_kv_insert(qkv, [1, 9, 2, 3], [0, 1, 40, -1], cs, cache, nkv)
    assert err == oracle.ERR_POSITION | oracle.ERR_SLOT
    assert np.array_equal(out[1], qkv[1])               # bad position: row untouched
    assert np.any(cache[0, 0, 0]) and not np.any(cache[0, 0, 1])   # slot 1 skipped
    assert not np.any(cache[1])                         # slot 40 out of range, -1 padding


# ---- the predecessor (layer front) -------------------------------------------

def test_layer_front_stream_is_exact_widening(oracle_lib):
    """stream = x as FP32: bf16 widening and fp32 copies are exact; aux = stream."""
    rng = np.random.default_rng(40)
    xb = _bf(rng.standard_normal((3, 256)) * 5).reshape(3, 256)
    stream, aux, _ = oracle.layer_front(xb, keep_aux=True)
    assert np.array_equal(stream.view(np.uint32), (xb.astype(np.uint32) << 16))
    assert np.array_equal(aux, stream)
    xf = rng.standard_normal((2, 256)).astype(np.float32)
    stream, aux, _ = oracle.layer_front(xf)
    assert np.array_equal(stream, xf) and aux is None


@pytest.mark.parametrize("c", [2.0 ** -10, 0.3, 7.0])
def test_layer_front_constant_row_closed_form(oracle_lib, c):
    """A constant row c with weight w: out = bf16(c / sqrt(c^2 + eps) * w) —
    a mean over the row (not a sum), eps inside the root, the weight applied."""
    hidden = 8192
    x = np.full((1, hidden), c, np.float32)
    w_vals = np.linspace(-2, 2, hidden).astype(np.float32)
    wb = _bf(w_vals)
    _, _, out = oracle.layer_front(x, wb)
    wf = wl.from_bits(wb).double().numpy()
    want = (c / math.sqrt(c * c + 1e-6)) * wf
    got = wl.from_bits(out).double().numpy()[0]
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-30)


def test_layer_front_rms_and_weight_linearity(oracle_lib):
    """Weightless rows come out with RMS 1 (to BF16 rounding); a weight of 2
    doubles every output exactly (power of two)."""
    rng = np.random.default_rng(41)
    x = (rng.standard_normal((4, 8192)) * 3).astype(np.float32)
    _, _, out1 = oracle.layer_front(x)
    v = wl.from_bits(out1).double().numpy()
    assert np.all(np.abs(np.sqrt(np.mean(v ** 2, axis=1)) - 1.0) < 4e-3)
    _, _, out2 = oracle.layer_front(x, _bf(np.full(8192, 2.0)))
    assert np.array_equal(wl.from_bits(out2).double().numpy(), 2 * v)


# ---- verify-step paged attention (attn2) -------------------------------------

def _torch_attn2(inp, nkv, window, scale, eps):
    """The same op through torch's scaled_dot_product_attention in float64
    (a library routine), gathering K and V through the block table."""
    qkv = inp["qkv"].double()
    cache = inp["kv_cache"].double()
    R = inp["context_lens"].shape[0]
    qh = 8 * nkv
    out = torch.empty(8 * R, qh * 64, dtype=torch.float64)
    gate0 = qh * 64 + 2 * nkv * 64
    for r in range(R):
        L = int(inp["context_lens"][r])
        pages = inp["block_table"][r, : (L + 15) // 16].long()
        kv = cache[pages].permute(1, 0, 2, 3).reshape(nkv, -1, 128)[:, :L]   # [nkv, L, 128]
        pos = torch.arange(L - 8, L)[:, None]
        j = torch.arange(L)[None, :]
        ok = j <= pos
        if window:
            ok &= j > pos - window
        for h in range(qh):
            q = qkv[8 * r: 8 * r + 8, h * 64:(h + 1) * 64]
            k, v = kv[h // 8, :, :64], kv[h // 8, :, 64:]
            o = torch.nn.functional.scaled_dot_product_attention(
                q[None], k[None], v[None], attn_mask=ok[None], scale=scale)[0]
            o = o / torch.sqrt(torch.mean(o * o, dim=1, keepdim=True) + eps)
            gt = qkv[8 * r: 8 * r + 8, gate0 + h * 64: gate0 + (h + 1) * 64]
            out[8 * r: 8 * r + 8, h * 64:(h + 1) * 64] = o * torch.sigmoid(gt)
    return out


@pytest.mark.parametrize("name", ["attn_r1_l8_nkv1", "attn_r3_mixed_nkv2"])
def test_attn2_matches_torch_sdpa(oracle_lib, name):
    w = wl.ATTN_WORKLOADS[name]
    inp = wl.make_attn_inputs(w)
    out, err = oracle.attn2(wl.bits(inp["qkv"]), wl.bits(inp["kv_cache"]), inp["block_table"].numpy(),
                            inp["context_lens"].numpy(), w.num_kv_heads, w.window)
    assert err == 0
    ref = _torch_attn2(inp, w.num_kv_heads, w.window, 0.125, 1e-6)
    got = wl.from_bits(out).double()
    assert torch.all((got - ref).abs() <= 2.0 ** -8 * ref.abs() + 1e-12)


def test_attn2_window_matches_torch_sdpa(oracle_lib):
    w = wl.AttnWorkload("win", R=2, num_kv_heads=1, context=(40, 100), num_pages=16, seed=77,
                        window=20)
    inp = wl.make_attn_inputs(w)
    out, err = oracle.attn2(wl.bits(inp["qkv"]), wl.bits(inp["kv_cache"]), inp["block_table"].numpy(),
                            inp["context_lens"].numpy(), 1, 20)
    ref = _torch_attn2(inp, 1, 20, 0.125, 1e-6)
    assert err == 0
    assert torch.all((wl.from_bits(out).double() - ref).abs() <= 2.0 ** -8 * ref.abs() + 1e-12)


def test_attn2_window_one_is_own_value(oracle_lib):
    """A window of 1 leaves each row its own key: o = V of position L-8+i, so
    out = bf16(norm(V) * sigmoid(gate)) (closed form, no softmax)."""
    w = wl.AttnWorkload("w1", R=1, num_kv_heads=1, context=(20,), num_pages=4, seed=78, window=1)
    inp = wl.make_attn_inputs(w)
    out, err = oracle.attn2(wl.bits(inp["qkv"]), wl.bits(inp["kv_cache"]), inp["block_table"].numpy(),
                            inp["context_lens"].numpy(), 1, 1)
    assert err == 0
    cache = inp["kv_cache"].double()
    for i in range(8):
        p = 12 + i
        page = int(inp["block_table"][0, p // 16])
        v = cache[page, 0, p % 16, 64:]
        o = v / torch.sqrt(torch.mean(v * v) + 1e-6)
        for h in range(8):
            gt = inp["qkv"][i, 512 + 128 + h * 64: 512 + 128 + (h + 1) * 64].double()
            want = (o * torch.sigmoid(gt)).float().to(torch.bfloat16)
            assert torch.equal(wl.from_bits(out[i, h * 64:(h + 1) * 64]), want)


def test_attn2_causal_and_page_remap(oracle_lib):
    """Keys after a row's position do not change it; moving the request's
    pages elsewhere in the cache (same contents) changes nothing."""
    w = wl.AttnWorkload("c", R=1, num_kv_heads=1, context=(50,), num_pages=16, seed=79)
    inp = wl.make_attn_inputs(w)
    args = (inp["block_table"].numpy(), inp["context_lens"].numpy(), 1)
    base, _ = oracle.attn2(wl.bits(inp["qkv"]), wl.bits(inp["kv_cache"]), *args)
    cache = wl.bits(inp["kv_cache"]).copy()
    last = 49
    pg = int(inp["block_table"][0, last // 16])
    cache[pg, 0, last % 16, :] ^= 0x0101                     # perturb key/value 49
    pert, _ = oracle.attn2(wl.bits(inp["qkv"]), cache, *args)
    assert np.array_equal(pert[:7], base[:7])                # rows 0..6 cannot see key 49
    assert not np.array_equal(pert[7], base[7])              # row 7 can
    table = inp["block_table"].numpy().copy()
    used = table[0, :4]
    free = np.setdiff1d(np.arange(16), used)[:4]
    moved = wl.bits(inp["kv_cache"]).copy()
    moved[free] = moved[used]
    table[0, :4] = free
    remap, _ = oracle.attn2(wl.bits(inp["qkv"]), moved, table, inp["context_lens"].numpy(), 1)
    assert np.array_equal(remap, base)


def test_attn2_bad_requests_are_skipped(oracle_lib):
    w = wl.AttnWorkload("bad", R=2, num_kv_heads=1, context=(20, 20), num_pages=8, seed=80)
    inp = wl.make_attn_inputs(w)
    lens = inp["context_lens"].numpy().copy()
    lens[0] = 5                                             # shorter than the 8 rows
    table = inp["block_table"].numpy().copy()
    table[1, 1] = 99                                        # page outside the cache
    start = np.full((16, 512), 0x1234, np.uint16)
    out, err = oracle.attn2(wl.bits(inp["qkv"]), wl.bits(inp["kv_cache"]), table, lens, 1,
                            out_bits=start)
    assert err == oracle.ERR_ATTN_REQUEST
    assert np.all(out == 0x1234)
