"""The C-ABI library: it loads, exports every symbol include/gla.h declares,
and rejects invalid arguments on the host before any launch. No GPU needed:
none of these calls reaches the device."""
import ctypes
import os
import re

import pytest

import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import binding as bnd
from chunkwise_gated_linear_gla_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return bnd.load()


def _declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        txt = open(os.path.join(ROOT, "include", h)).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        names += re.findall(r"\b(gla_\w+)\s*\(", txt)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert "gla_fwd" in declared and "gla_fwd_ex" in declared
    for n in declared:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(declared) <= set(bnd.EXPORTED) | set(declared)
    for n in bnd.EXPORTED:
        assert n in declared, f"binding wraps {n}, which include/ does not declare"


def test_struct_layout_matches_header():
    # 7 pointers, 8 ints, pointer, size_t, 2 ints, pointer, int (+ 4 bytes of tail padding)
    assert ctypes.sizeof(bnd.gla_fwd_params) == 7 * 8 + 8 * 4 + 8 + 8 + 2 * 4 + 8 + 4 + 4
    assert bnd.gla_fwd_params.workspace.offset == 88
    assert bnd.gla_fwd_params.log_b.offset == 112
    assert bnd.gla_fwd_params.window_chunks.offset == 120


def test_plain_c_client_sees_the_binding_layout(lib, tmp_path):
    """include/gla.h compiles as C99 and links against libgla.so; the parameter structs
    have the layout the Python binding declares."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    build = os.path.dirname(bnd.library_path())
    exe = str(tmp_path / "abi_client")
    cmd = [cc, "-std=c99", "-Wall", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
           os.path.join(ROOT, "tests", "csrc", "abi_client.c"), "-L", build, "-lgla", "-Wl,-rpath," + build,
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    fwd = [int(x) for x in out[0].split()[1:]]
    bwd = [int(x) for x in out[1].split()[1:]]
    F, Bw = bnd.gla_fwd_params, bnd.gla_bwd_params
    assert fwd == [ctypes.sizeof(F), F.workspace.offset, F.path.offset, F.log_b.offset, F.window_chunks.offset]
    assert bwd == [ctypes.sizeof(Bw), Bw.workspace.offset, Bw.path.offset, Bw.log_b.offset, Bw.grad_log_b.offset]
    assert out[2].startswith("status GLA_ERR_INVALID_ARG")
    assert int(out[3].split()[1]) == gla.gla_version()


def test_status_strings(lib):
    for s in range(6):
        txt = gla.gla_status_string(s)
        assert txt.startswith("GLA_")
    assert gla.gla_version() >= 100


def _params(**kw):
    p = bnd.gla_fwd_params()
    base = dict(q=0x10000, k=0x20000, v=0x30000, log_g=0x40000, S0=None, O=0x50000, ST=None,
                B=1, H=1, T=64, dk=64, dv=64, chunk=64, dtype=bnd.GLA_BF16,
                gate=bnd.GLA_GATE_PER_KEY, workspace=None, workspace_bytes=0,
                force_segments=0, path=bnd.GLA_PATH_AUTO)
    base.update(kw)
    for k, v in base.items():
        setattr(p, k, v)
    return p


BAD = [
    ("null q", dict(q=None), bnd.GLA_ERR_INVALID_ARG),
    ("null O", dict(O=None), bnd.GLA_ERR_INVALID_ARG),
    ("B=0", dict(B=0), bnd.GLA_ERR_INVALID_ARG),
    ("H<0", dict(H=-1), bnd.GLA_ERR_INVALID_ARG),
    ("T<0", dict(T=-5), bnd.GLA_ERR_INVALID_ARG),
    ("dk not /16", dict(dk=40), bnd.GLA_ERR_INVALID_ARG),
    ("dv not /16", dict(dv=72 + 1), bnd.GLA_ERR_INVALID_ARG),
    ("gate none with log_g", dict(gate=bnd.GLA_GATE_NONE), bnd.GLA_ERR_INVALID_ARG),
    ("per-key gate without log_g", dict(log_g=None), bnd.GLA_ERR_INVALID_ARG),
    ("misaligned q", dict(q=0x10002), bnd.GLA_ERR_INVALID_ARG),
    ("misaligned O", dict(O=0x50008), bnd.GLA_ERR_INVALID_ARG),
    ("O overlaps v", dict(O=0x30000 + 64), bnd.GLA_ERR_INVALID_ARG),
    ("ST overlaps k", dict(ST=0x20000), bnd.GLA_ERR_INVALID_ARG),
    ("ST partially overlaps S0", dict(S0=0x100000, ST=0x100000 + 256), bnd.GLA_ERR_INVALID_ARG),
    ("bad dtype", dict(dtype=7), bnd.GLA_ERR_INVALID_ARG),
    ("bad gate", dict(gate=9), bnd.GLA_ERR_INVALID_ARG),
    ("bad path", dict(path=5), bnd.GLA_ERR_INVALID_ARG),
    ("negative segments", dict(force_segments=-1), bnd.GLA_ERR_INVALID_ARG),
    ("misaligned workspace", dict(workspace=0x7000010, workspace_bytes=1 << 20), bnd.GLA_ERR_INVALID_ARG),
    ("bilinear gate without log_b", dict(gate=4), bnd.GLA_ERR_INVALID_ARG),
    ("log_b with the per-key gate", dict(log_b=0x900000), bnd.GLA_ERR_INVALID_ARG),
    ("log_b overlaps O", dict(gate=4, log_b=0x50000 + 16), bnd.GLA_ERR_INVALID_ARG),
    ("tensor path with the bilinear gate in fp32",
     dict(gate=4, log_b=0x900000, dtype=bnd.GLA_FP32, dv=128, path=bnd.GLA_PATH_TENSOR), bnd.GLA_ERR_UNSUPPORTED),
    ("chunk 32", dict(chunk=32), bnd.GLA_ERR_UNSUPPORTED),
    ("dk 784", dict(dk=784), bnd.GLA_ERR_UNSUPPORTED),
    ("tensor path with dk 384", dict(dk=384, path=bnd.GLA_PATH_TENSOR, q=0x1000000, k=0x9000000, v=0x11000000,
                                     log_g=0x21000000, O=0x31000000), bnd.GLA_ERR_UNSUPPORTED),
    ("tensor path with fp32", dict(dtype=bnd.GLA_FP32, path=bnd.GLA_PATH_TENSOR), bnd.GLA_ERR_UNSUPPORTED),
    ("tensor path with dv 48", dict(dv=48, path=bnd.GLA_PATH_TENSOR), bnd.GLA_ERR_UNSUPPORTED),
]


@pytest.mark.parametrize("name,kw,want", BAD, ids=[b[0] for b in BAD])
def test_rejects_before_launch(lib, name, kw, want):
    p = _params(**kw)
    assert bnd.gla_fwd_ex(p, stream=0, check=False) == want
    assert bnd.gla_fwd_stage(p, 0, stream=0, check=False) == want
    assert bnd.gla_fwd_num_stages(p) == -1
    assert bnd.gla_fwd_workspace_size(p) == 0


def test_gla_fwd_rejects_before_launch(lib):
    # gla_fwd's signature: dk not a multiple of 16
    s = bnd.gla_fwd(0x10000, 0x20000, 0x30000, 0x40000, None, 0x50000, None, 1, 1, 64, 40, 64, 64,
                    stream=0, check=False)
    assert s == bnd.GLA_ERR_INVALID_ARG
    s = bnd.gla_fwd(0x10000, 0x20000, 0x30000, None, None, 0x50000, None, 1, 1, 64, 64, 64, 128,
                    stream=0, check=False)
    assert s == bnd.GLA_ERR_UNSUPPORTED


def test_plan_on_host():
    # in-place state carry (ST == S0) is valid
    p = _params(S0=0x100000, ST=0x100000)
    assert bnd.gla_fwd_num_stages(p) >= 1
    # bf16 with supported shapes plans the tensor path: prep + chunk pass, with workspace
    p = _params(dk=256, dv=512, T=2048, B=8, H=4, q=0x1000000, k=0x9000000, v=0x11000000,
                log_g=0x21000000, O=0x31000000)
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
    assert names == ["gla_chunk_prep", "gla_chunk_fwd"]
    assert bnd.gla_fwd_workspace_size(p) > 0
    # the fused per-key pass on request: one kernel, no workspace, never a sequence split
    p.path = bnd.GLA_PATH_FUSED
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
    assert names == ["gla_chunk_fused"]
    assert bnd.gla_fwd_workspace_size(p) == 0
    p.force_segments = 4
    assert [bnd.gla_fwd_stage_name(p, 0)] == ["gla_chunk_fused"]
    # shapes and gates it does not take
    for kw in (dict(dk=128), dict(dv=1024), dict(gate=bnd.GLA_GATE_TOKEN_SCALAR), dict(dtype=bnd.GLA_FP32)):
        q = _params(dk=256, dv=512, T=2048, B=8, H=4, q=0x1000000, k=0x9000000, v=0x11000000,
                    log_g=0x21000000, O=0x31000000, path=bnd.GLA_PATH_FUSED)
        for key, val in kw.items():
            setattr(q, key, val)
        assert bnd.gla_fwd_num_stages(q) == -1 and bnd.gla_fwd_ex(q, stream=0, check=False) == bnd.GLA_ERR_UNSUPPORTED
    p = _params(dk=256, dv=512, T=2048, B=8, H=4, q=0x1000000, k=0x9000000, v=0x11000000,
                log_g=0x21000000, O=0x31000000)
    # forced segments add the state pass and the scan
    p.force_segments = 4
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
    assert names == ["gla_chunk_prep", "gla_chunk_state", "gla_state_scan", "gla_chunk_fwd"]
    ws_exact = bnd.gla_fwd_workspace_size(p)
    # the sliding-window split (opt-in) replaces the state pass and the scan with one window
    # pass, which writes the 4 segments' start states directly; the exact split also keeps
    # the 3 pieces' states of its state pass (one piece per segment here: 3 x 128 pieces
    # would not fit in one wave) and one more start state
    p.window_chunks = 4
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
    assert names == ["gla_chunk_prep", "gla_chunk_state_window", "gla_chunk_fwd"]
    assert bnd.gla_fwd_workspace_size(p) == ws_exact - 3 * 32 * 256 * 512 * 4
    # without a split the window changes nothing
    p.force_segments = 1
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
    assert names == ["gla_chunk_prep", "gla_chunk_fwd"]
    p.window_chunks = -1
    assert bnd.gla_fwd_num_stages(p) == -1 and bnd.gla_fwd_ex(p, stream=0, check=False) == bnd.GLA_ERR_INVALID_ARG
    p.window_chunks = 0
    # fp32 takes the CUDA-core path, no workspace
    p = _params(dtype=bnd.GLA_FP32)
    assert [bnd.gla_fwd_stage_name(p, 0)] == ["gla_fwd_simt"]
    assert bnd.gla_fwd_workspace_size(p) == 0
    # empty sequence: only the state copy
    p = _params(T=0, q=None, k=None, v=None, O=None)
    assert bnd.gla_fwd_stage_name(p, 0) == "gla_copy_state"
    # keys wider than 256 (up to 768) take the CUDA-core path in bf16 too, except dk = 512
    for dk in (272, 384, 768):
        p = _params(dk=dk, dv=1024, q=0x1000000, k=0x9000000, v=0x11000000, log_g=0x21000000, O=0x31000000)
        assert bnd.gla_fwd_num_stages(p) == 1 and bnd.gla_fwd_stage_name(p, 0) == "gla_fwd_simt"
        assert bnd.gla_fwd_workspace_size(p) == 0
    # dk = 512: the tensor path in two key halves, never split along the sequence; the
    # workspace holds the first half's fp32 output
    p = _params(dk=512, dv=1024, T=2048, B=8, H=2, q=0x100000000, k=0x200000000, v=0x300000000,
                log_g=0x400000000, O=0x500000000, force_segments=0)
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
    assert names == ["gla_chunk_prep", "gla_chunk_fwd", "gla_chunk_fwd_keys_hi"]
    assert bnd.gla_fwd_workspace_size(p) >= 8 * 2 * 2048 * 1024 * 4
    p.force_segments = 4
    assert [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))] == names
    p.gate, p.log_b = bnd.GLA_GATE_BILINEAR, 0x600000000
    assert [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))] == ["gla_fwd_simt"]


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(bnd, "_lib", None)
    monkeypatch.setattr(bnd._build, "LIB", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="not built"):
        bnd.load()


def test_bench_segment_rule_matches_library_plan():
    """bench.py mirrors the library's split rule to count bytes; the workspace the library
    plans (one fp32 state per state-pass piece, and one start state per piece plus the
    last segment's) must agree with it."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from chunkwise_gated_linear_gla_gb300 import inputs as gi
    for name in ("linear_attn", "scalar_decay", "gla_1p3b", "gla_long"):
        w = gi.WORKLOADS[name]
        p = _params(B=w.B, H=w.H, T=w.T, dk=w.dk, dv=w.dv, gate=w.gate,
                    log_g=None if w.gate == 0 else 0x40000000, q=0x100000000, k=0x200000000,
                    v=0x300000000, O=0x400000000)
        # the library plans for 148 SMs without a device
        nseg, cps, sub, st_nseg, st_cps = bench.planned_split(w, 0, 148)
        assert st_nseg == (nseg - 1) * sub and st_cps * sub == (cps if nseg > 1 else 0), name
        BH = w.B * w.H
        nch = (w.T + 63) // 64
        # Q (.) Lambda and K (.) Gamma and the chunk decays with a gate; the score tiles unless
        # the chunk pass forms every chunk's scores itself (no gate, dk <= 128)
        sc_all = bench.scores_in_chunk_pass(w) and w.gate == 0
        base = (0 if w.gate == 0 else 2 * BH * nch * 64 * w.dk * 2 + BH * nch * w.dk * 4) + \
            (0 if sc_all else BH * nch * 64 * 64 * 2)
        seg = BH * (2 * st_nseg + 1) * w.dk * w.dv * 4 if nseg > 1 else 0
        assert bnd.gla_fwd_workspace_size(p) == got_staged(p), name
        got = bnd.gla_fwd_workspace_size(p)
        assert abs(got - (base + seg)) < 4096, (name, got, base + seg, nseg)


def test_plan_scores_in_chunk_pass():
    """dk <= 128 without a gate: the chunk pass forms the intra-chunk scores itself, so there is
    no prep stage and, without a split, no workspace; the per-head decay keeps its prep (for
    K (.) Gamma, and the steep chunks' scores); dk = 256 or a per-key gate keep the score tiles."""
    kw = dict(B=8, H=16, T=2048, dk=128, dv=128, q=0x1000000, k=0x9000000, v=0x11000000,
              O=0x31000000, gate=bnd.GLA_GATE_NONE, log_g=None)
    p = _params(**kw)
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
    assert names == ["gla_chunk_fwd"] and bnd.gla_fwd_workspace_size(p) == 0
    p.force_segments = 2   # only the split's states
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
    assert names == ["gla_chunk_state", "gla_state_scan", "gla_chunk_fwd"]
    assert bnd.gla_fwd_workspace_size(p) == 128 * (1 + 1 + 1) * 128 * 128 * 4
    p = _params(**dict(kw, dk=256))
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
    assert names == ["gla_chunk_prep", "gla_chunk_fwd"]
    assert bnd.gla_fwd_workspace_size(p) == 128 * 32 * 64 * 64 * 2
    p = _params(**dict(kw, gate=bnd.GLA_GATE_HEAD_SCALAR, log_g=0x21000000))
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
    assert names == ["gla_chunk_prep", "gla_chunk_fwd"]
    # dk = 64 without a gate: the chunk pass alone as well; the per-token and per-key gates
    # (whose scores need the prep's per-row or per-key factors) keep the prep at dk <= 128
    p = _params(**dict(kw, dk=64))
    assert [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))] == ["gla_chunk_fwd"]
    assert bnd.gla_fwd_workspace_size(p) == 0
    for g in (bnd.GLA_GATE_TOKEN_SCALAR, bnd.GLA_GATE_PER_KEY):
        p = _params(**dict(kw, gate=g, log_g=0x21000000))
        names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
        assert names == ["gla_chunk_prep", "gla_chunk_fwd"], (g, names)


def test_split_rule_over_random_shapes():
    """The library's sequence-split plan (segments, state-pass pieces) and its score placement
    against bench.py's mirror of the rule, over seeded random shapes, gates and forced segment
    counts, through the workspace size: the per-gate tiles, plus one fp32 state per piece and
    one start state per piece and after the last."""
    import random
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from chunkwise_gated_linear_gla_gb300 import inputs as gi
    rnd = random.Random(5)
    gates = [(bnd.GLA_GATE_NONE, 0), (bnd.GLA_GATE_HEAD_SCALAR, 1), (bnd.GLA_GATE_PER_KEY, 2),
             (bnd.GLA_GATE_TOKEN_SCALAR, 3)]
    for _ in range(300):
        gate, g = rnd.choice(gates)
        B, H = rnd.choice([1, 2, 3]), rnd.choice([1, 2, 4, 8])
        dk, dv = rnd.choice([64, 128, 256]), 128 * rnd.choice([1, 2, 4])
        T = rnd.randint(1, 64 * 300)
        force = rnd.choice([0, 0, 1, 2, 3, 5, 9, 17])
        ng = {0: None, 1: 0x2000000000, 2: 0x2000000000, 3: 0x2000000000}[g]
        p = _params(B=B, H=H, T=T, dk=dk, dv=dv, gate=gate, log_g=ng, q=0x100000000, k=0x400000000,
                    v=0x800000000, O=0xC00000000, force_segments=force)
        w = gi.Workload("t", B=B, H=H, T=T, dk=dk, dv=dv, dtype=gi.WORKLOADS["gla_1p3b"].dtype, gate=g)
        nseg, cps, sub, st_nseg, st_cps = bench.planned_split(w, force, 148)
        BH, nch = B * H, (T + 63) // 64
        sc_all = bench.scores_in_chunk_pass(w) and g == 0
        base = (0 if g == 0 else 2 * BH * nch * 64 * dk * 2 + BH * nch * dk * 4) + \
            (0 if sc_all else BH * nch * 64 * 64 * 2)
        seg = BH * (2 * st_nseg + 1) * dk * dv * 4 if nseg > 1 else 0
        got = bnd.gla_fwd_workspace_size(p)
        assert abs(got - (base + seg)) < 4 * 256, (B, H, T, dk, dv, g, force, got, base + seg, nseg, sub)
        names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
        assert ("gla_chunk_prep" in names) == (not sc_all), names
        assert ("gla_chunk_state" in names) == (nseg > 1), (names, nseg)


def got_staged(p):
    q = bnd.gla_fwd_params.from_buffer_copy(p)
    q.path = bnd.GLA_PATH_STAGED
    return bnd.gla_fwd_workspace_size(q)


def test_plan_bilinear_on_host():
    """The bilinear gate on the tensor path: key prep, value prep, chunk pass, then the CUDA-core
    pass for flagged heads; never a sequence split; the workspace adds V (.) D' (bf16), the
    chunks' column decays and one flag per head."""
    kw = dict(B=1, H=2, T=65536, dk=256, dv=512, q=0x1000000, k=0x11000000, v=0x21000000,
              log_g=0x31000000, O=0x41000000, gate=4, log_b=0x61000000)
    p = _params(**kw)
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]
    assert names == ["gla_chunk_prep", "gla_value_prep", "gla_chunk_fwd", "gla_fwd_simt_flagged"]
    # the per-key gate on the same shapes splits the sequence (2 heads x 4 dv tiles)
    pk = _params(**dict(kw, gate=bnd.GLA_GATE_PER_KEY, log_b=None))
    names_pk = [bnd.gla_fwd_stage_name(pk, i) for i in range(bnd.gla_fwd_num_stages(pk))]
    assert "gla_chunk_state" in names_pk
    BH, T, dk, dv, nch = 2, 65536, 256, 512, 1024
    base = 2 * BH * T * dk * 2 + BH * nch * 64 * 64 * 2 + BH * nch * dk * 4
    extra = BH * T * dv * 2 + BH * nch * dv * 4 + 256
    assert bnd.gla_fwd_workspace_size(p) == base + extra


def test_segment_pair_plan_on_host(lib):
    """Workspace of the sequence-exchange pair: the tensor route's gate-prep workspace (one
    segment) plus the log gate's fp64 partial sums; the CUDA-core route's discarded O."""
    BH, T, dk, dv = 4, 300, 128, 256
    nch = (T + 63) // 64
    big = dict(q=0x1000000, k=0x9000000, v=0x11000000, log_g=0x21000000, O=None,
               B=2, H=2, T=T, dk=dk, dv=dv)
    prep = 2 * BH * nch * 64 * dk * 2 + BH * nch * 64 * 64 * 2 + BH * nch * dk * 4
    sums = -(-(1 * BH * dk * 8) // 256) * 256            # one 1024-token slice
    assert bnd.gla_segment_pair_workspace_size(_params(**big)) == prep + sums
    # no q: the pair does not need it
    assert bnd.gla_segment_pair_workspace_size(_params(**dict(big, q=None))) == prep + sums
    # fp32 inputs: the CUDA-core pass, O to the workspace
    o32 = BH * T * dv * 4
    assert bnd.gla_segment_pair_workspace_size(_params(**dict(big, dtype=bnd.GLA_FP32))) == o32 + sums
    # per-head scalar gate: no partial sums; bilinear gate: not supported (0); T = 0: nothing
    hs = bnd.gla_segment_pair_workspace_size(_params(**dict(big, gate=bnd.GLA_GATE_HEAD_SCALAR)))
    assert hs == prep
    assert bnd.gla_segment_pair_workspace_size(_params(**dict(big, gate=bnd.GLA_GATE_BILINEAR,
                                                              log_b=0x41000000))) == 0
    assert bnd.gla_segment_pair_workspace_size(_params(**dict(big, T=0))) == 0


def test_segment_pair_and_scan_reject_before_launch(lib):
    p = _params(q=0x1000000, k=0x9000000, v=0x11000000, log_g=0x21000000, O=None, B=1, H=2, T=64, dk=128, dv=128)
    G, S = 0x31000000, 0x41000000
    assert bnd.gla_segment_pair(p, G, None, stream=0, check=False) == bnd.GLA_ERR_INVALID_ARG
    assert bnd.gla_segment_pair(p, S, S, stream=0, check=False) == bnd.GLA_ERR_INVALID_ARG    # aliased outputs
    assert bnd.gla_segment_pair(p, G, 0x9000000, stream=0, check=False) == bnd.GLA_ERR_INVALID_ARG  # S* over k
    pb = _params(gate=bnd.GLA_GATE_BILINEAR, log_b=0x900000)
    assert bnd.gla_segment_pair(pb, G, S, stream=0, check=False) == bnd.GLA_ERR_UNSUPPORTED
    sc = lambda *a: bnd.gla_pair_scan(*a, stream=0, check=False)
    dims = (1, 2, 128, 128)
    ns = 2 * 128 * 128 * 4
    assert sc(-1, G, S, None, 0x51000000, None, *dims) == bnd.GLA_ERR_INVALID_ARG        # P < 0
    assert sc(2, G, S, None, None, None, *dims) == bnd.GLA_ERR_INVALID_ARG               # no output
    assert sc(2, None, S, None, 0x51000000, None, *dims) == bnd.GLA_ERR_INVALID_ARG      # pairs missing
    assert sc(2, G, S, None, S + ns, None, *dims) == bnd.GLA_ERR_INVALID_ARG             # S_in inside S*
    assert sc(1, G, S, 0x61000000, None, 0x61000000 + 64, *dims) == bnd.GLA_ERR_INVALID_ARG  # S_T over S0
    cb = lambda *a: bnd.gla_pair_combine(*a, 1, 2, 128, 128, stream=0, check=False)
    assert cb(G, S, G, 0x51000000) == bnd.GLA_ERR_INVALID_ARG                            # pair 1 aliases pair 2
    assert cb(G, S, 0x51000000, 0x51000000 + 64) == bnd.GLA_ERR_INVALID_ARG              # log Gamma1 inside S1


def test_selftest_wait_limit_checked_before_launch(lib):
    assert bnd.gla_selftest_bounded_wait(0, stream=0, check=False) == bnd.GLA_ERR_INVALID_ARG
    assert bnd.gla_selftest_bounded_wait(1000001, stream=0, check=False) == bnd.GLA_ERR_INVALID_ARG
