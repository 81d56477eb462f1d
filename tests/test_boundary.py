"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every function include/qkvfront.h declares, and refuses bad calls on the host
before any CUDA call."""
import ctypes
import os
import re

import pytest
import torch

from kv_insert_gb300 import qkv_front as qf
from kv_insert_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return qf.load()


def test_library_exports_every_declared_function(lib):
    names = qf.header_functions()
    assert len(names) >= 10
    raw = ctypes.CDLL(qf.library_path())
    for n in names:
        assert hasattr(raw, n), n


def test_binding_uses_only_declared_functions():
    src = open(os.path.join(ROOT, "kv_insert_gb300", "qkv_front.py")).read()
    used = set(re.findall(r"lib\.(qkv_front\w*)", src)) | set(re.findall(r"load\(\)\.(qkv_front\w*)", src))
    assert used <= set(qf.header_functions()), used - set(qf.header_functions())


def test_strerror_every_code(lib):
    for code in range(0, 10):
        assert qf.strerror(code)
    assert "unknown" in qf.strerror(99)


# fake, 16-byte aligned addresses: the checks below fail before anything is read
X, W, POS, SL, CS, OUT, CACHE = ((i + 1) << 36 for i in range(7))


def call(lib, x=X, w=W, pos=POS, sl=SL, cs=CS, rows=4096, out=OUT, cache=CACHE, pages=4, M=1,
         N=1152, nkv=1):
    return lib.qkv_front(x, w, pos, sl, cs, rows, out, cache, pages, M, N, nkv, None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=17), 1), (dict(M=-1), 1),
    (dict(N=1153), 2), (dict(nkv=0), 2), (dict(N=2304, nkv=1), 2),
    (dict(x=0), 3), (dict(cache=0), 3), (dict(pos=0), 3),
    (dict(x=X + 2), 4), (dict(w=W + 8), 4), (dict(out=OUT + 4), 4), (dict(sl=SL + 4), 4),
    (dict(rows=0), 7), (dict(pages=0), 7),
    (dict(out=X), 9), (dict(cache=W + 64), 9),
])
def test_host_refusals_before_any_cuda_call(lib, kw, code):
    assert call(lib, **kw) == code
    args = dict(x=X, w=W, pos=POS, sl=SL, cs=CS, rows=4096, out=OUT, cache=CACHE, pages=4, M=1,
                N=1152, nkv=1)
    args.update(kw)
    why = lib.qkv_front_unsupported(args["x"], args["w"], args["pos"], args["sl"], args["cs"],
                                    args["rows"], args["out"], args["cache"], args["pages"],
                                    args["M"], args["N"], args["nkv"])
    assert why is not None and len(why) > 5


def test_zero_tokens_is_a_no_op(lib):
    assert call(lib, M=0, x=0, out=0) == 0


def test_variant_and_launch_variant_refusals(lib):
    assert lib.qkv_front_variant(1152, 0, None, None, None, None, None) == 1
    assert lib.qkv_front_variant(1000, 4, None, None, None, None, None) == 2
    lv = lib.qkv_front_launch_variant
    assert lv(X, W, POS, SL, CS, 4096, OUT, CACHE, 4, 1, 1152, 1, 3, 4, 0, 0, None) == 8  # splits 3
    assert lv(X, W, POS, SL, CS, 4096, OUT, CACHE, 4, 1, 1152, 1, 1, 1, 0, 0, None) == 8  # 1 stage
    assert lv(X, W, POS, SL, CS, 4096, OUT, CACHE, 4, 1, 1152, 1, 1, 3, 3, 0, None) == 8  # kb 3
    assert lv(X, W, POS, SL, CS, 4096, OUT, CACHE, 4, 1, 1152, 1, 1, 3, 0, 7, None) == 8  # consumer
    assert lv(X, W, POS, SL, CS, 4096, OUT, CACHE, 4, 1, 1152, 1, 1, 40, 4, 0, None) == 8  # smem
    assert lib.qkv_front_set_wait_limit(5) == 9
    assert lib.qkv_front_selftest_wait(0, None) == 9
    assert lib.qkv_front_prepare(1000, 1) == 2


def test_no_gpu_here_is_reported_not_crashed(lib):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid arguments: the call reaches the device query, which fails cleanly
    assert call(lib) in (5, 6)


def test_layout_helpers():
    q = torch.zeros(3, 9216)
    qv, gv = qf.split_qkv(q, 8)
    assert qv.shape == (3, 4096) and gv.shape == (3, 4096)
    assert gv.data_ptr() == q.data_ptr() + (4096 + 1024) * 4
    with pytest.raises(ValueError):
        qf.split_qkv(q, 4)
    assert qf.supports_shape(1152, 1) and qf.supports_shape(18432, 16)
    assert not qf.supports_shape(1152, 2)
    assert [qf.token_tiles(m) for m in (1, 8, 9, 16)] == [1, 1, 2, 2]


def test_product_path_never_touches_the_oracle():
    """The library and its binding share no code with the oracle and never
    import, link or run it."""
    pkg = os.path.join(ROOT, "kv_insert_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "qkv_oracle" not in text and "liboracle" not in text, f


def test_variants_the_gpu_tests_launch_are_accepted(lib):
    """Every (splits, stages) the GPU tests request passes the host-side
    variant check: the call gets past it to the device query (which fails on
    a machine without a GPU) instead of returning QKVF_ERR_VARIANT."""
    if torch.cuda.is_available():
        pytest.skip("checked through the GPU tests themselves")
    import test_determinism as td
    from kv_insert_gb300 import workloads as wl
    cases = [(n, s, st) for n, _ in [("m8_nkv8_n9216", 0), ("m16_nkv8_n9216_consecutive", 0),
                                   ("m1_nkv1_n1152", 0)] for s in (1, 2, 8)
             for st in td.RING_DEPTHS]
    cases += [(n, s, td.split_stages(s)) for n, sl in td.SPLIT_CASES for s in sl]
    cases += [(n, s, 3) for n, sl in td.SPLIT_CASES for s in sl]
    for name, splits, stages in cases:
        w = wl.WORKLOADS[name]
        for consumer in (0, 1, 2):
            for kb in (0, 1, 2, 4):
                rc = lib.qkv_front_launch_variant(X, W, POS, SL, CS, 4096, OUT, CACHE, 4, w.M, w.N,
                                                  w.num_kv_heads, splits, stages, kb, consumer,
                                                  None)
                assert rc in (5, 6), (name, splits, stages, kb, consumer, rc)


def test_resident_engine_variant_rule(lib):
    """The resident engine runs only at its fixed shape (8 CTAs per head, kb
    4, 4 stages): other explicit shapes are refused on the host, the fixed
    one gets past the check to the device query."""
    lv = lib.qkv_front_launch_variant
    args = (X, W, POS, SL, CS, 4096, OUT, CACHE, 4, 1, 1152, 1)
    assert lv(*args, 8, 4, 4, 3, None) in (5, 6)
    assert lv(*args, 8, 4, 0, 3, None) in (5, 6)
    assert lv(*args, 4, 4, 4, 3, None) == 8
    assert lv(*args, 8, 3, 4, 3, None) == 8
    assert lv(*args, 8, 4, 2, 3, None) == 8
    assert lv(*args, 8, 4, 4, 4, None) == 8   # no such engine


def test_from_host_refusals(lib):
    fh = lib.qkv_front_from_host
    need = lib.qkv_front_staging_bytes(8, 9216)
    assert need >= 8 * 8192 * 2 + 8 * 9216 * 2 + 2 * 64
    assert need % 256 == 0
    args = lambda st=OUT, nbytes=need, M=8: (X, POS, SL, CACHE + (1 << 35), W, CS, 4096, CACHE, 4096,
                                             st, nbytes, M, 9216, 8, None)
    assert fh(*args(M=17)) == 1
    assert fh(*args(M=0)) == 0
    assert fh(*args(st=OUT + 16)) == 4          # staging not 256-byte aligned
    assert fh(*args(nbytes=need - 256)) == 7    # staging too small
    assert lib.qkv_front_staging_bytes(17, 9216) == 0


def test_standalone_epilogue_refusals(lib):
    f = lib.qknorm_rope_kv_insert
    base = dict(qkv=X, pos=POS, sl=SL, cs=CS, rows=4096, cache=CACHE, pages=64, T=100, N=9216, nkv=8)

    def call(**kw):
        a = dict(base, **kw)
        return f(a["qkv"], a["pos"], a["sl"], a["cs"], a["rows"], a["cache"], a["pages"], a["T"],
                 a["N"], a["nkv"], None)
    assert call(T=-1) == 1 and call(T=(1 << 24) + 1) == 1
    assert call(N=1152) == 2 and call(nkv=0) == 2
    assert call(qkv=0) == 3 and call(sl=0) == 3
    assert call(qkv=X + 4) == 4 and call(pos=POS + 4) == 4
    assert call(rows=0) == 7 and call(pages=0) == 7
    assert call(cs=X + 128) == 9                     # table inside qkv
    assert call(T=0, qkv=0) == 0
    assert call() in (5, 6)                          # valid: reaches the device query
    why = lib.qknorm_rope_kv_insert_unsupported(X, POS, SL, CS, 4096, CACHE, 64, 100, 1152, 8)
    assert why is not None and b"1152" in why


def test_layer_front_refusals(lib):
    f = lib.layer_front
    ok = dict(x=X, f32=0, w=0, s=SL, a=0, o=OUT, rows=8, eps=1e-6)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["x"], a["f32"], a["w"] or None, a["s"], a["a"] or None, a["o"], a["rows"],
                 a["eps"], None)
    assert call(rows=-1) == 1 and call(rows=(1 << 20) + 1) == 1
    assert call(f32=2) == 9 and call(eps=0.0) == 9 and call(eps=-1.0) == 9
    assert call(x=0) == 3 and call(o=0) == 3
    assert call(x=X + 8) == 4 and call(a=CACHE + 4) == 4
    assert call(o=SL + 64) == 9            # out inside stream
    assert call(a=SL) == 9                 # aux is stream
    assert call(rows=0, x=0) == 0
    assert call() in (5, 6)                # valid: reaches the device query


def test_set_pdl_refusals(lib):
    assert lib.qkv_front_set_pdl(2) == 9 and lib.qkv_front_set_pdl(-1) == 9
    assert lib.qkv_front_set_pdl(0) == 0 and lib.qkv_front_set_pdl(1) == 0


def test_attn2_refusals(lib):
    f = lib.attn2
    ok = dict(q=X, c=CACHE, pages=64, bt=POS, mb=8, cl=SL, R=2, N=2304, nkv=2, win=0, sc=0.125,
              eps=1e-6, out=OUT)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["c"], a["pages"], a["bt"], a["mb"], a["cl"], a["R"], a["N"], a["nkv"],
                 a["win"], a["sc"], a["eps"], a["out"], None)
    assert call(R=-1) == 1 and call(R=65536) == 1
    assert call(N=1152) == 2 and call(nkv=0) == 2
    assert call(pages=0) == 7 and call(mb=0) == 7
    assert call(win=-1) == 9 and call(sc=0.0) == 9 and call(eps=2.0) == 9
    assert call(q=0) == 3 and call(bt=0) == 3
    assert call(q=X + 8) == 4 and call(cl=SL + 2) == 4
    assert call(out=X) == 9                           # out on top of qkv
    assert call(R=0, q=0) == 0
    assert call() in (5, 6)
    assert lib.attn2_launch_splits(X, CACHE, 64, POS, 8, SL, 2, 2304, 2, 0, 0.125, 1e-6, OUT, 3,
                                   None) == 8


def test_attn2_split_kv_refusals(lib):
    """The workspace checks come before any device query: a missing,
    misaligned, short or overlapping workspace and a bad split are refused."""
    WS = 1 << 44
    need = lib.attn2_split_kv_workspace_bytes(2, 2, 3)
    assert need == 2 * 2 * 3 * 17152                # one slot per (request, KV head, split)
    assert lib.attn2_split_kv_workspace_bytes(1, 1, 1) == 17152
    assert lib.attn2_split_kv_workspace_bytes(0, 2, 3) == 0
    assert lib.attn2_split_kv_workspace_bytes(1, 1, 257) == 0
    assert lib.attn2_split_kv_workspace_bytes(1, 65, 1) == 0
    ok = dict(q=X, c=CACHE, pages=64, bt=POS, mb=8, cl=SL, R=2, N=2304, nkv=2, win=0, sc=0.125,
              eps=1e-6, out=OUT, S=3, ws=WS, n=need)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.attn2_split_kv(a["q"], a["c"], a["pages"], a["bt"], a["mb"], a["cl"], a["R"], a["N"],
                                  a["nkv"], a["win"], a["sc"], a["eps"], a["out"], a["S"], a["ws"],
                                  a["n"], None)
    assert call(R=-1) == 1 and call(N=1152) == 2 and call(q=0) == 3
    assert call(S=-1) == 8 and call(S=257) == 8
    assert call(ws=0) == 3
    assert call(ws=WS + 16) == 4
    assert call(n=need - 1) == 7
    assert call(ws=OUT) == 9                         # workspace on top of out
    assert call(ws=CACHE) == 9                       # workspace inside the cache
    assert call(R=0, ws=0) == 0
    assert call() in (5, 6)                          # valid: reaches the device query


def test_unsupported_projection_reasons():
    """The host-side refusals of a projection layer the front cannot take
    (no device needed)."""
    w = torch.zeros(2304, 8192, dtype=torch.bfloat16)
    assert qf.unsupported_projection(w) is None
    assert "quantized" in qf.unsupported_projection(w, quantized=True)
    assert "float16" in qf.unsupported_projection(w.to(torch.float16))
    assert "bias" in qf.unsupported_projection(w, bias=torch.zeros(2304))
    assert "neox" in qf.unsupported_projection(w, is_neox_style=True)
    assert "gathered" in qf.unsupported_projection(w, gather_output=True)
    assert "cos" in qf.unsupported_projection(w, cos_sin=torch.zeros(16, 64, dtype=torch.float16))
    assert qf.unsupported_projection(w, cos_sin=torch.zeros(16, 64)) is None
    assert "1152" in qf.unsupported_projection(torch.zeros(2000, 8192, dtype=torch.bfloat16))
    assert "shape" in qf.unsupported_projection(torch.zeros(2304, 4096, dtype=torch.bfloat16))


def test_attn2_unsupported_reasons(lib):
    """The C ABI's attn2_unsupported gives the reason of each host refusal
    (NULL only past the checks, at the device query, which has no GPU here)."""
    f = lib.attn2_unsupported
    ok = dict(q=X, c=CACHE, pages=64, bt=POS, mb=8, cl=SL, R=2, N=2304, nkv=2, win=0, sc=0.125,
              eps=1e-6, out=OUT)

    def why(**kw):
        a = dict(ok, **kw)
        r = f(a["q"], a["c"], a["pages"], a["bt"], a["mb"], a["cl"], a["R"], a["N"], a["nkv"],
              a["win"], a["sc"], a["eps"], a["out"])
        return None if r is None else r.decode()
    assert "num_reqs" in why(R=-1)
    assert "1152" in why(N=1152)
    assert "num_kv_heads" in why(nkv=0)
    assert "window" in why(win=-1)
    assert "scale" in why(sc=0.0) and "eps" in why(eps=2.0) and "eps" in why(eps=0.0)
    assert "NULL" in why(q=0)
    assert "aligned" in why(q=X + 8)
    assert "overlaps" in why(out=X)
    # past every check the device query answers (no GB300 here)
    assert why() in ("a CUDA call failed", "the current GPU is not compute capability 10.3 (sm_103a)")


def test_unsupported_attn2_layer_reasons():
    """The binding's layer check (page cute_ops, unsupported_attn2): a layer
    without the o-norm and sigmoid gate, another head_dim or q / KV ratio, and
    a scale or eps outside what the kernel takes are refused."""
    from types import SimpleNamespace as L
    base = dict(use_o_norm=True, use_o_gate=True, head_dim=64, num_heads=64, num_kv_heads=8,
                scaling=0.125, rms_norm_eps=1e-6)
    assert qf.unsupported_attn2(L(**base)) is None
    assert "gate" in qf.unsupported_attn2(L(**dict(base, use_o_gate=False)))
    assert "norm" in qf.unsupported_attn2(L(**dict(base, use_o_norm=False)))
    assert "128 dims" in qf.unsupported_attn2(L(**dict(base, head_dim=128)))
    assert "q heads" in qf.unsupported_attn2(L(**dict(base, num_heads=32)))
    assert "scale" in qf.unsupported_attn2(L(**dict(base, scaling=0.0)))
    assert "eps" in qf.unsupported_attn2(L(**dict(base, rms_norm_eps=0.0)))
    assert qf.unsupported_attn2(L(**dict(base, scaling=0.0883883))) is None


def test_noalloc_refusals_without_a_device(lib):
    """Above one split the 256-slot bound is checked before any device query;
    at one split (no slots used) the same shape gets past it."""
    f = lib.attn2_split_kv_noalloc
    args = (X, CACHE, 256, POS, 8, SL, 40, 9216, 8, 0, 0.125, 1e-6, OUT)
    assert f(*args, 2, None) == 7        # 40 x 8 x 2 = 640 slots > 256
    assert f(*args, 1, None) in (5, 6)   # one split: reaches the device query
