"""GPU backward element by element against the rounding model (tight check).

The fp64-oracle comparison in test_gpu_bwd.py has to leave room for the
kernels' bf16 roundings of P, dS and the certified forward's O, which alone
move dQ by up to 4% of its largest entry.  Here both sides start from the same
O and lse2 -- those of tests/rounding_model.py's certified forward, computed on
the CPU -- and the GPU's dQ, dK, dV are compared with the model's backward,
which applies the kernels' own roundings; the bound (gpu_util.TIGHT_TOL)
leaves room for fp32 accumulation order only.

The populations are the ones the oracle bounds were derived on: 320 short
causal heads (where a row dominated by one key gives the certified forward's
rounded weight to D_i and so to dK: the effect a GPU run once showed at 1.5e-2
of max |dK| against the oracle) and diffuse DiT heads (dQ's cancellation of
the shared key bias).  For those, the test also checks that the GPU's error
against the exact oracle is the model's own error against it: the whole gap
to the oracle is the rounding the model describes.
"""
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
import rounding_model as rm
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, make_dout, make_inputs
from gpu_util import assert_grads_tight, grad_errors, need_gpu, report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    oracle.set_num_threads(os.cpu_count() or 1)
    clis.clis_clear_device_error()
    yield


@pytest.fixture(autouse=True)
def _device_error_word_stays_clear():
    yield
    code = clis.clis_get_device_error()
    clis.clis_clear_device_error()
    assert code == 0, f"device error word {code:#x}"


POPULATIONS = [
    # workload recipe, B, H, N, seed
    ("causal", 8, 40, 300, 61),   # 320 short causal heads
    ("causal", 1, 32, 512, 62),
    ("480p", 1, 32, 1024, 63),    # diffuse DiT heads
    ("causal", 1, 4, 1500, 64),   # several tiles with a ragged tail
    ("tiny", 1, 8, 700, 65),      # d = 64, non-causal
]


@pytest.mark.parametrize("name,B,H,N,seed", POPULATIONS)
def test_backward_matches_rounding_model(name, B, H, N, seed):
    dev = need_gpu()
    w = dataclasses.replace(WORKLOADS[name], B=B)
    q, k, v = make_inputs(w, device=dev, N=N, H=H, seed=seed)
    do = make_dout(q.shape, device=dev, seed=seed)
    scale = w.softmax_scale()
    qf, kf, vf, gf = (t.reshape(-1, N, w.d).double().cpu().numpy() for t in (q, k, v, do))
    BH = qf.shape[0]
    o_m = np.empty_like(qf)
    lse2_m = np.empty((BH, N))
    for h in range(BH):
        o_m[h], lse2_m[h] = rm.certified_forward(qf[h], kf[h], vf[h], scale, w.causal)
    o = torch.from_numpy(o_m).reshape(q.shape).to(torch.bfloat16).to(dev)
    lse2 = torch.from_numpy(lse2_m.astype(np.float32)).reshape(-1).to(dev)
    dq, dk, dv = clis.attention_bwd(q, k, v, o, do, lse2, causal=w.causal)
    torch.cuda.synchronize()
    got = [t.reshape(BH, N, w.d).float().cpu().numpy() for t in (dq, dk, dv)]
    model = [np.empty_like(qf) for _ in range(3)]
    for h in range(BH):
        for i, x in enumerate(rm.backward(qf[h], kf[h], vf[h], o_m[h], gf[h], lse2_m[h], scale, w.causal)):
            model[i][h] = x
    what = f"bwd tight {name} {B}x{H}x{N}"
    for g, m, n in zip(got, model, ("dq", "dk", "dv")):
        assert_grads_tight(g, m, n, what)
    if N > 1024:
        return
    # Against the exact oracle: the GPU's worst error per gradient is the
    # model's own (the same rounding), to within the tight bound.
    ref = oracle.attention_bwd(*(t.reshape(-1, N, w.d).cpu() for t in (q, k, v, do)), scale, causal=w.causal)
    for g, m, r, n in zip(got, model, ref, ("dq", "dk", "dv")):
        e_gpu = grad_errors(g, r)[0].max()
        e_model = grad_errors(rm.bf16(m), r)[0].max()
        report(f"{what} {n} vs oracle", gpu=float(e_gpu), model=float(e_model))
        assert abs(e_gpu - e_model) <= 1e-2, (n, e_gpu, e_model)
