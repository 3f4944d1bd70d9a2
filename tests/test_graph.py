"""The forward pass captured into a CUDA graph and replayed (the launch sequence
of gla_fwd_ex, including the chunk pass's programmatic dependent launch, needs
no host work per replay): every replay on new inputs written into the captured
buffers matches the fp64 oracle."""
import pytest
import torch

import oracle
import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import binding as bnd
from chunkwise_gated_linear_gla_gb300 import build as gbuild
from chunkwise_gated_linear_gla_gb300 import inputs as gi

from _util import assert_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


@pytest.mark.parametrize("path,segments", [(gla.GLA_PATH_STAGED, 0), (gla.GLA_PATH_STAGED, 3),
                                           (gla.GLA_PATH_FUSED, 0)], ids=["staged", "split", "fused"])
def test_forward_replays_from_a_cuda_graph(path, segments):
    w = gi.Workload("t", B=1, H=2, T=300, dk=256, dv=512, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.1)
    x0 = gi.make_inputs(w, seed=120)
    buf = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x0.items()}
    O = torch.empty(w.B, w.H, w.T, w.dv, dtype=torch.bfloat16, device="cuda")
    ST = torch.empty(w.B, w.H, w.dk, w.dv, device="cuda")
    p = bnd.make_params(buf["q"], buf["k"], buf["v"], buf["log_g"], buf["S0"], O, ST, path=path,
                        force_segments=segments)
    nb = bnd.gla_fwd_workspace_size(p)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    if nb:
        p.workspace, p.workspace_bytes = ws.data_ptr(), nb
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        bnd.gla_fwd_ex(p, s)   # one eager call first (per-device set-up outside the capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        bnd.gla_fwd_ex(p, s)
    torch.cuda.synchronize()
    for seed in (121, 122, 123):
        x = gi.make_inputs(w, seed=seed)
        for k in ("q", "k", "v", "log_g", "S0"):
            buf[k].copy_(x[k])
        O.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert gla.gla_device_status() == 0
        Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
        assert_close(to_np(O), Oref, torch.bfloat16, f"O (replay, seed {seed})")
        assert_close(to_np(ST), STref, torch.bfloat16, f"ST (replay, seed {seed})")
