"""The seeded input generators (no GPU needed): determinism, the permutation
structure of perm (whole, and in independent blocks), bf16 storage, routing
weights, and the hc_post coefficient shapes."""
import pytest
import torch

from gen import CONFIGS, make_inputs, make_mhc_inputs


def _is_bf16_exact(x):
    return torch.equal(x.float().to(torch.bfloat16).float(), x.float())


@pytest.mark.parametrize("kind", ["random", "expert_sorted"])
@pytest.mark.parametrize("blocks", [1, 2, 4])
def test_perm_is_a_permutation_within_each_block(kind, blocks):
    T = 8
    inp = make_inputs("dsv3_decode", T, seed=3, perm_kind=kind, perm_blocks=blocks)
    K = inp["K"]
    p = inp["perm"].reshape(blocks, -1)
    per = T * K // blocks
    for b in range(blocks):
        assert sorted(p[b].tolist()) == list(range(b * per, (b + 1) * per))


def test_expert_sorted_single_block_is_the_whole_sort_and_differs_from_random():
    a = make_inputs("dsv3_decode", 16, seed=9, perm_kind="expert_sorted")
    b = make_inputs("dsv3_decode", 16, seed=9, perm_kind="random")
    assert not torch.equal(a["perm"], b["perm"])
    # the same routing draw either way: weights identical
    assert torch.equal(a["w"], b["w"])


def test_draws_are_seeded():
    a = make_inputs("glm_gemma", 4, seed=5)
    b = make_inputs("glm_gemma", 4, seed=5)
    c = make_inputs("glm_gemma", 4, seed=6)
    for key in ("perm", "w", "residual", "gamma"):
        assert torch.equal(a[key], b[key])
    assert all(torch.equal(x, y) for x, y in zip(a["E"], b["E"]))
    assert not torch.equal(a["residual"], c["residual"])


@pytest.mark.parametrize("name", list(CONFIGS))
def test_config_inputs_have_the_stated_shapes_and_types(name):
    cfg = CONFIGS[name]
    T = min(cfg.Ts)
    inp = make_inputs(name, T)
    R, K, H = cfg.R, cfg.K, cfg.H
    assert inp["residual"].dtype == torch.bfloat16 and inp["residual"].shape == (T, H)
    assert inp["gamma"].dtype == torch.bfloat16 and inp["gamma"].shape == (H,)
    g = inp["gamma"].float()
    assert bool(((g >= 0.5) & (g <= 1.5)).all())
    if K > 0:
        assert len(inp["E"]) == R and all(e.shape == (T * K, H) and e.dtype == torch.bfloat16 for e in inp["E"])
        assert inp["perm"].dtype == torch.int32 and inp["perm"].shape == (T, K)
        assert inp["w"].dtype == torch.float32 and inp["w"].shape == (T, K)
        # softmax / renormalised top-k: positive weights summing to 1 per token
        assert bool((inp["w"] > 0).all())
        assert torch.allclose(inp["w"].sum(1), torch.ones(T), atol=1e-5)
    if inp["S"] is not None:
        assert len(inp["S"]) == R and all(s.shape == (T, H) for s in inp["S"])


def test_mhc_inputs():
    m = make_mhc_inputs(4, 264, 4, 5, seed=1)
    assert len(m["P"]) == 4 and m["x"].shape == (5, 4, 264)
    assert all(_is_bf16_exact(p) for p in m["P"]) and _is_bf16_exact(m["x"])
    post = m["post"]
    assert bool(((post > 0) & (post < 2)).all())
    comb = m["comb"].double()
    assert bool((comb > 0).all())
    # doubly stochastic to the precision of 20 alternating normalisations
    assert torch.allclose(comb.sum(2), torch.ones(5, 4, dtype=torch.float64), atol=1e-5)
    assert torch.allclose(comb.sum(1), torch.ones(5, 4, dtype=torch.float64), atol=1e-5)
