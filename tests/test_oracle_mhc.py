"""Pins of the all-reduce + mHC write-back (hc_post) oracle (CPU only).

PARITY UNPINNED against the pages: sglang PR #42020 (Summary, Scope) says only
that hc_post reads the all-reduced FFN output back and mixes it into the four
residual streams.  The reading the oracle implements,

    out[t,i,j] = post[t,i] * sum_r P_r[t,j] + sum_k comb[t,i,k] * x[t,k,j],

is pinned here against an exact rational brute force, its special cases
(identity mix, pure all-reduce, single stream = residual add, which the main
oracle computes independently) and its symmetries.  None of these can show
that the reading is the pages' own.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from oracle.brute import brute_ar_mhc_post
from gen import bf16_bits, make_mhc_inputs


def _np(inp):
    P = [bf16_bits(p) for p in inp["P"]]
    x = bf16_bits(inp["x"])
    return P, x, inp["post"].numpy(), inp["comb"].numpy()


@pytest.mark.parametrize("R,hc", [(1, 1), (2, 2), (2, 4), (3, 4)])
def test_mhc_brute_force(R, hc):
    inp = make_mhc_inputs(R, 8, hc, 2, seed=11 + R + hc)
    P, x, post, comb = _np(inp)
    got = oracle.ar_mhc_post_ref(P, x, post, comb)
    exact = brute_ar_mhc_post([p.tolist() for p in P], x.tolist(), post.tolist(), comb.tolist())
    for t, i, j in itertools.product(range(2), range(hc), range(8)):
        e = float(exact[t][i][j])
        assert abs(got[t, i, j] - e) <= 1e-12 * max(1.0, abs(e)), (t, i, j, got[t, i, j], e)


def test_mhc_identity_mix_returns_the_streams():
    inp = make_mhc_inputs(4, 64, 4, 3)
    P, x, post, comb = _np(inp)
    out = oracle.ar_mhc_post_ref(P, x, np.zeros_like(post), np.broadcast_to(np.eye(4, dtype=np.float32), comb.shape))
    ref = inp["x"].double().numpy()
    assert np.array_equal(out, ref)


def test_mhc_pure_all_reduce_matches_the_main_oracle():
    """comb = 0, post = 1: every output stream is the all-reduce, which the main
    oracle (K = 0, zero residual) computes on its own code path."""
    inp = make_mhc_inputs(4, 64, 4, 3)
    P, x, post, comb = _np(inp)
    out = oracle.ar_mhc_post_ref(P, x, np.ones_like(post), np.zeros_like(comb))
    zero = np.zeros((3, 64), np.uint16)
    h = oracle.ar_rmsnorm_ref(P, zero, np.full(64, 0x3F80, np.uint16), 0.0, 1e-6)["h"]
    for i in range(4):
        assert np.array_equal(out[:, i], h)


def test_mhc_single_stream_is_the_residual_add():
    """hc = 1, post = 1, comb = 1: the write-back is y + x, the residual add the
    main oracle performs before its norm."""
    inp = make_mhc_inputs(2, 96, 1, 5)
    P, x, post, comb = _np(inp)
    out = oracle.ar_mhc_post_ref(P, x, np.ones_like(post), np.ones_like(comb))
    h = oracle.ar_rmsnorm_ref(P, x[:, 0, :], np.full(96, 0x3F80, np.uint16), 0.0, 1e-6)["h"]
    assert np.array_equal(out[:, 0], h)


def test_mhc_stream_relabelling():
    inp = make_mhc_inputs(3, 32, 4, 2)
    P, x, post, comb = _np(inp)
    base = oracle.ar_mhc_post_ref(P, x, post, comb)
    sigma = [2, 0, 3, 1]
    # relabel the incoming streams: the same mix, summed in another order
    out = oracle.ar_mhc_post_ref(P, np.ascontiguousarray(x[:, sigma]), post,
                                 np.ascontiguousarray(comb[:, :, sigma]))
    assert np.allclose(out, base, rtol=1e-13, atol=1e-13)
    # relabel the outgoing streams: the outputs permute, bit for bit
    out = oracle.ar_mhc_post_ref(P, x, np.ascontiguousarray(post[:, sigma]),
                                 np.ascontiguousarray(comb[:, sigma, :]))
    assert np.array_equal(out, base[:, sigma])


def test_mhc_scales_with_its_inputs():
    """Doubling every partial and stream doubles every output exactly."""
    inp = make_mhc_inputs(2, 48, 4, 2)
    P, x, post, comb = _np(inp)
    base = oracle.ar_mhc_post_ref(P, x, post, comb)
    dbl = lambda t: bf16_bits((t.float() * 2).to(torch.bfloat16))
    out = oracle.ar_mhc_post_ref([dbl(p) for p in inp["P"]], dbl(inp["x"]), post, comb)
    assert np.array_equal(out, 2 * base)


def test_mhc_hand_example():
    """hc = 2, one token, one column, worked by hand: P = (1, 2) so y = 3;
    x = (4, -8); post = (0.5, 2); comb = [[1, 0.25], [0.5, 0]]:
    out_0 = 0.5*3 + 1*4 + 0.25*(-8) = 3.5;  out_1 = 2*3 + 0.5*4 + 0 = 8."""
    bits = lambda v: np.array(v, np.float32).view(np.uint32).__rshift__(16).astype(np.uint16)
    P = [bits([[1.0]]), bits([[2.0]])]
    x = bits([[[4.0], [-8.0]]])
    out = oracle.ar_mhc_post_ref(P, x, np.array([[0.5, 2.0]], np.float32),
                                 np.array([[[1.0, 0.25], [0.5, 0.0]]], np.float32))
    assert out.tolist() == [[[3.5], [8.0]]]
