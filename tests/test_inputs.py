"""The seeded synthetic inputs match their stated recipe (CPU only).

Every workload draws x, B, C ~ N(0, 1) (B, C scaled by 1/sqrt(N) for the
bf16 workloads), dt = softplus(N(mu, 0.5)), A = -exp(U(0, ln 16)) per head,
D ~ N(0, 1) per head and, where the workload has them, initial states
~ N(0, 0.1^2); shapes and dtypes follow the workload, and a seed gives the
same tensors every time.  The statistics are checked on the first 2048
tokens of one sequence, enough for tight bounds.
"""
import math

import pytest
import torch

from state_space_model_gb300 import inputs as gen


def _small(w):
    return w.with_(batch=1, seqlen=min(w.seqlen, 2048))


@pytest.mark.parametrize("name", sorted(gen.WORKLOADS))
def test_shapes_dtypes_and_layout(name):
    w = _small(gen.WORKLOADS[name])
    d = gen.make_inputs(w)
    Bn, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    st = torch.float32 if w.dtype == "f32" else torch.bfloat16
    want = {"x": ((Bn, L, H, P), st), "dt": ((Bn, L, H), torch.float32),
            "A": ((H,), torch.float32), "B": ((Bn, L, G, N), st),
            "C": ((Bn, L, G, N), st), "D": ((H,), torch.float32)}
    for k, (shape, dtype) in want.items():
        assert tuple(d[k].shape) == shape and d[k].dtype == dtype, k
        assert d[k].is_contiguous(), k
    if w.init_states:
        assert tuple(d["initial_states"].shape) == (Bn, H, P, N)
        assert d["initial_states"].dtype == torch.float32
    else:
        assert d["initial_states"] is None


@pytest.mark.parametrize("name", sorted(gen.WORKLOADS))
def test_distributions(name):
    w = _small(gen.WORKLOADS[name])
    d = gen.make_inputs(w)
    f = lambda k: d[k].double()
    assert abs(f("x").mean().item()) < 0.02 and abs(f("x").std().item() - 1.0) < 0.02
    bc_std = 1.0 / math.sqrt(w.dstate) if w.dtype == "bf16" else 1.0
    for k in ("B", "C"):
        assert abs(f(k).std().item() / bc_std - 1.0) < 0.05, k
    # dt = softplus(z), z ~ N(mu, 0.5): invert the softplus and check z
    dt = f("dt")
    assert (dt > 0).all()
    z = torch.log(torch.expm1(dt))
    assert abs(z.mean().item() - w.dt_mu) < 0.02 and abs(z.std().item() - 0.5) < 0.02
    A = f("A")
    assert ((A <= -1.0) & (A >= -16.0)).all()
    # log(-A) ~ U(0, ln 16): every value inside, the heads spread over it
    u = torch.log(-A) / math.log(16.0)
    assert u.min().item() >= 0.0 and u.max().item() <= 1.0
    if w.nheads >= 24:
        assert u.min().item() < 0.25 and u.max().item() > 0.75
    if w.init_states:
        assert abs(f("initial_states").std().item() - 0.1) < 0.005


def test_same_seed_same_tensors_and_seeds_differ():
    w = _small(gen.WORKLOADS["mamba2_2p7b"]).with_(seqlen=256)
    a, b = gen.make_inputs(w), gen.make_inputs(w)
    c = gen.make_inputs(w, seed=w.seed + 1)
    for k in ("x", "dt", "A", "B", "C", "D"):
        assert torch.equal(a[k], b[k]), k
        assert not torch.equal(a[k], c[k]), k


def test_workload_seeds_follow_the_recipe():
    order = ["tiny_f32", "mamba2_130m", "mamba2_2p7b", "hybrid_g8", "long_64k"]
    assert [gen.WORKLOADS[n].seed for n in order] == [20261, 20262, 20263, 20264, 20265]
    assert gen.WORKLOADS["long_64k"].dt_mu == -3.0
    assert all(gen.WORKLOADS[n].dt_mu == -2.0 for n in order[:4])
