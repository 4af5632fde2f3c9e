"""GPU parity of the gated delta-rule decode step (Gated DeltaNet / KDA) against the fp64
oracle, through the C ABI.

Bar (float32 arithmetic): each state entry within 64 float32 ulps of 1 + max|S| and each
output within 64 ulps of max|o| + max|S| * sum|q|: the kernel rounds the fade, a dot product
of dk terms (dk/32 per lane, then a 32-lane tree), the correction and the read, each a
few ulps of the magnitudes involved.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24


@pytest.fixture(scope="module")
def kvd():
    import kv_cache_decode_split_gb300 as m
    return m


def _gpu_step(kvd, x):
    S = x.S.clone().cuda()
    o = kvd.delta_decode_step(S, x.q.cuda(), x.k.cuda(), x.v.cuda(), x.a.cuda(), x.beta.cuda())
    torch.cuda.synchronize()
    return S.cpu().double().numpy(), o.cpu().double().numpy()


def _check(S_gpu, o_gpu, S_ref, o_ref, q):
    tol_S = 64 * U32 * (1 + np.abs(S_ref).max())
    tol_o = 64 * U32 * (np.abs(o_ref).max() + np.abs(S_ref).max() * np.abs(q).sum(-1).max())
    assert np.abs(S_gpu - S_ref).max() <= tol_S, (np.abs(S_gpu - S_ref).max(), tol_S)
    assert np.abs(o_gpu - o_ref).max() <= tol_o, (np.abs(o_gpu - o_ref).max(), tol_o)


@pytest.mark.parametrize("dk", [64, 128, 256])
@pytest.mark.parametrize("dv", [128, 40, 8, 1])
@pytest.mark.parametrize("per_channel", [True, False])
def test_delta_step_small(kvd, dk, dv, per_channel):
    n = 37
    x = W.make_delta(n, dk, dv, per_channel=per_channel, seed=7000 + dk + dv, state_factor=1.0)
    S_gpu, o_gpu = _gpu_step(kvd, x)
    S_ref, o_ref = oracle.delta_step(x.S, x.q, x.k, x.v, x.a, x.beta)
    _check(S_gpu, o_gpu, S_ref, o_ref, x.q.numpy())


def test_delta_step_single_head(kvd):
    x = W.make_delta(1, 128, 128, seed=7100)
    S_gpu, o_gpu = _gpu_step(kvd, x)
    S_ref, o_ref = oracle.delta_step(x.S, x.q, x.k, x.v, x.a, x.beta)
    _check(S_gpu, o_gpu, S_ref, o_ref, x.q.numpy())


def test_delta_step_full_size(kvd):
    # the benchmark's workload, every head checked
    x = W.build("kda_decode")
    S_gpu, o_gpu = _gpu_step(kvd, x)
    S_ref, o_ref = oracle.delta_step(x.S, x.q, x.k, x.v, x.a, x.beta)
    _check(S_gpu, o_gpu, S_ref, o_ref, x.q.numpy())


def test_delta_steps_carry_state_in_place(kvd):
    # twenty tokens in a row: the state stays on the device and is updated in place; the
    # oracle carries its own fp64 state from the same start with the same per-token inputs
    n, T = 16, 20
    x0 = W.make_delta(n, 128, 128, seed=7200, state_factor=0.5)
    S = x0.S.clone().cuda()
    S_ref = x0.S.double().numpy()
    for t in range(T):
        xt = W.make_delta(n, 128, 128, seed=7300 + 10 * t)
        o = kvd.delta_decode_step(S, xt.q.cuda(), xt.k.cuda(), xt.v.cuda(), xt.a.cuda(),
                                  xt.beta.cuda())
        S_ref, o_ref = _oracle_fp64_state(S_ref, xt)
    torch.cuda.synchronize()
    err = np.abs(S.cpu().double().numpy() - S_ref).max()
    assert err <= T * 64 * U32 * (1 + np.abs(S_ref).max()), err
    assert np.abs(o.cpu().double().numpy() - o_ref).max() <= T * 64 * U32 * (1 + np.abs(o_ref).max())


def _oracle_fp64_state(S_ref, x):
    # the oracle reads a float32 state; its fp64 state is passed as the nearest float32 and
    # the rounding it drops is added back, which the step carries linearly (fade, write,
    # read are linear in S for fixed inputs)
    S32 = S_ref.astype(np.float32)
    lo = S_ref - S32.astype(np.float64)
    S_new, o = oracle.delta_step(S32, x.q, x.k, x.v, x.a, x.beta)
    zero = np.zeros_like(x.v.numpy())
    dS, do = oracle.delta_step(lo.astype(np.float32), x.q, x.k, zero, x.a, x.beta)
    return S_new + dS, o + do


def test_delta_step_rejects_bad_arguments(kvd):
    x = W.make_delta(2, 128, 128, seed=7400)
    S = x.S.clone().cuda()
    q, k, v, a, b = (t.cuda() for t in (x.q, x.k, x.v, x.a, x.beta))
    # unsupported key width
    S96 = torch.zeros(2, 128, 96, device="cuda")
    with pytest.raises(kvd.KvdError) as e:
        kvd.delta_decode_step(S96, torch.zeros(2, 96, device="cuda"),
                              torch.zeros(2, 96, device="cuda"), v, torch.ones(2, device="cuda"), b)
    assert e.value.status == -2
    # the output may not overlap the state
    with pytest.raises(kvd.KvdError) as e:
        kvd.delta_decode_step(S, q, k, v, a, b, o=S.view(-1)[:256].view(2, 128))
    assert e.value.status == -1
    # a state that is not 16-byte aligned
    buf = torch.zeros(2 * 128 * 128 + 1, device="cuda")
    with pytest.raises(kvd.KvdError) as e:
        kvd.delta_decode_step(buf[1:].view(2, 128, 128), q, k, v, a, b)
    assert e.value.status == -1
