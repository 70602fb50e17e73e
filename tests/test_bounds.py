"""The element-wise rounding bound used for the stress backward (CPU only).

tests.parity.backward_rounding_bounds claims a first-order bound on the error
of a backward that rounds O, P, dS and its outputs to a 16-bit type.  Here a
CPU emulation of exactly those roundings (fp64 elsewhere) must stay inside
the bound, and a result with a localised mistake must not.
"""
import torch

import oracle
from seeded_inputs import Workload, make_inputs
from tests.parity import backward_rounding_bounds


def _emulate_16bit_backward(q, k, v, do, causal, scale, dt):
    """fp64 arithmetic with the kernels' four roundings to dt: stored O, P and dS operands, outputs."""
    q, k, v, do = (oracle.as_f64(x) for x in (q, k, v, do))
    rnd = lambda x: x.to(dt).to(torch.float64)  # noqa: E731
    p, _ = oracle.softmax_rows(oracle.scores(q, k, scale, causal))
    o_stored = rnd(p @ v)
    delta = (do * o_stored).sum(-1, keepdim=True)
    dp = do @ v.transpose(-1, -2)
    ds = rnd(p * (dp - delta))
    dq = rnd(scale * ds @ k)
    dk = rnd(scale * ds.transpose(-1, -2) @ q)
    dv = rnd(rnd(p).transpose(-1, -2) @ do)
    return dq, dk, dv


def _case(qk_std, dtype, causal, S=384, D=64, seed=5):
    w = Workload("bound", 1, 1, S, D, dtype, causal, qk_std=qk_std, backward=True, seed=seed)
    inp = make_inputs(w)
    args = [inp[n][0, 0] for n in ("q", "k", "v", "do")]
    return w, args


def test_emulated_16bit_backward_is_inside_the_bound():
    for qk_std, dtype, causal in ((2.0, "bf16", False), (1.0, "bf16", True), (2.0, "fp16", False),
                                  (1.0, "fp16", True)):
        w, args = _case(qk_std, dtype, causal)
        u = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -11
        exact = oracle.backward(*args, causal, w.scale)
        emu = _emulate_16bit_backward(*args, causal, w.scale, w.torch_dtype)
        bounds = backward_rounding_bounds(*args, causal, w.scale, u=u)
        for name, e, r, b in zip(("dQ", "dK", "dV"), emu, exact, bounds):
            ratio = float(((e - r).abs() / b).max())
            assert ratio <= 0.5, f"{dtype} std {qk_std} causal {causal} {name}: {ratio:.2f} of the bound"


def test_localised_mistake_exceeds_the_bound():
    """One wrong row or a dropped scale factor is caught element by element."""
    w, args = _case(2.0, "bf16", False)
    exact = oracle.backward(*args, False, w.scale)
    bq, bk, bv = backward_rounding_bounds(*args, False, w.scale, u=2.0 ** -8)
    bad = exact[0].clone()
    bad[17] += 0.05  # one row off by 0.05
    assert float(((bad - exact[0]).abs() / bq).max()) > 1.0
    bad_dk = exact[1] * 1.05  # dK off by 5 %
    assert float(((bad_dk - exact[1]).abs() / bk).max()) > 1.0
    q, k, v, do = args
    shifted = oracle.backward(q, k, v, torch.roll(do, 1, 0), False, w.scale)[2]  # dV from misaligned dO rows
    assert float(((shifted - exact[2]).abs() / bv).max()) > 1.0
