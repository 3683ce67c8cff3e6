"""qmoe_ffn (the MoE feed-forward layer) against the oracle, through the C ABI.

Every output of the config-4 layer (128 experts, d_model 2048, d_ff 768,
top-8, Q4_0) at 1, 8 and 64 tokens, within the tolerance the per-product bar
implies through SwiGLU and the down projection (oracle/moe.py); plus the
refusals and the bad-expert latch.
"""
import numpy as np
import pytest

from gemv_mul_mm_gb300 import synth
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    import torch  # noqa: F401
    from gemv_mul_mm_gb300 import build as qbuild
    from gemv_mul_mm_gb300 import qmm
    qbuild.build()
    qmm.set_path(0)
    return qmm


def layer(Q, p, ids=None, **kw):
    ids = p["ids"] if ids is None else ids
    return Q.qmoe_ffn(p["kind"], dev(p["w_gu"]), p["gu_stride"], dev(p["w_down"]), p["down_stride"],
                      p["n_experts"], dev(p["x"]), dev(ids), dev(p["w"]), p["d_model"], p["d_ff"], **kw)


@pytest.mark.parametrize("T", synth.MOE["tokens"])
def test_moe_layer_matches_oracle(Q, orc, T):
    import torch
    p = synth.moe_layer_problem(T)
    Y = torch.full((T, p["d_model"]), -1e30, dtype=torch.float32, device="cuda")
    layer(Q, p, Y=Y)
    assert Q.last_path() == Q.PATH_MOE
    assert Q.check_device_error() == 0
    got = Y.cpu().numpy().astype(np.float64)
    assert not np.any(got == -1e30)
    y, tol = orc.moe_ffn(p["kind"], p["w_gu"], p["gu_stride"], p["w_down"], p["down_stride"], p["n_experts"],
                         p["x"], p["ids"], p["w"], p["d_model"], p["d_ff"], nthreads=8)
    bad = ~(np.abs(got - y) <= tol)
    assert not bad.any(), f"{int(bad.sum())} of {got.size} outputs outside the derived tolerance"


def test_moe_layer_bad_expert_and_refusals(Q):
    import torch
    p = synth.moe_layer_problem(2)
    ids = p["ids"].copy()
    ids[1, 3] = 999                                  # token 1 routed to a missing expert
    Y = layer(Q, p, ids=ids)
    assert Q.check_device_error() == Q.STATUS_ID["QMM_ERR_BAD_EXPERT_ID"]
    got = Y.cpu().numpy()
    assert np.all(np.isnan(got[1])) and np.all(np.isfinite(got[0]))
    # a workspace one byte short is refused before anything runs
    need = Q.qmoe_ffn_workspace_bytes(2, 8, p["d_model"], p["d_ff"])
    ws = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(Q.QmmError) as e:
        layer(Q, p, workspace=ws)
    assert e.value.name == "QMM_ERR_WORKSPACE_TOO_SMALL"
