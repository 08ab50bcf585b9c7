"""Pins of the oracle's router (scoring, correction bias, top-k) against what
the definition and arithmetic fix, independent of the oracle's own loops.

The router's reading (sigmoid scores, selection on score + bf16 correction
bias, K need not be a power of two, equal keys: lower expert first, weights
renormalised over the picks and scaled) is stated in oracle/moe_oracle.c."""
import numpy as np
import pytest
import torch

import oracle


def _bf16(a):
    return torch.as_tensor(a, dtype=torch.float32).to(torch.bfloat16)


def test_zero_input_selects_by_bias_alone_with_equal_weights():
    """x = 0: every logit is 0, every score 1/2, so the keys are 1/2 + bias: the
    picks are the experts of largest bias (equal biases: lower index first) and
    the renormalised weights are scale / K each (closed form)."""
    E, K, H = 12, 6, 32
    bias = _bf16([0.5, -1, 0.25, 0.5, 0, 3, 0.25, -2, 0.5, 1, 0.25, 0.125])
    x = torch.zeros(2, H, dtype=torch.bfloat16)
    wr = _bf16(np.random.default_rng(0).standard_normal((E, H)))
    ids, w, keys = oracle.route(x, wr, bias, 2, H, E, K, scale=2.5, renorm=True)
    # bias descending, ties by index: 5 (3), 9 (1), 0, 3, 8 (0.5), 2 (0.25) -- 6 and 10 tie with 2 but come later
    assert ids.tolist() == [[5, 9, 0, 3, 8, 2]] * 2
    assert np.allclose(w, np.full((2, K), 2.5 / K), rtol=1e-15, atol=0)  # scale * (1/2) / (K/2)
    assert np.array_equal(keys[0], 0.5 + bias.double().numpy())


def test_without_renorm_weights_are_scaled_scores():
    E, K, H = 8, 3, 16
    x = torch.zeros(1, H, dtype=torch.bfloat16)
    wr = torch.zeros(E, H, dtype=torch.bfloat16)
    ids, w, _ = oracle.route(x, wr, None, 1, H, E, K, scale=2.0, renorm=False)
    assert ids.tolist() == [[0, 1, 2]]  # all keys equal: lowest indices, in order
    assert np.array_equal(w, np.full((1, K), 1.0))  # 2.0 * sigmoid(0)


def test_exact_ties_go_to_the_lower_expert_brute_force():
    """Exhaustive over every bias pattern on a 4-level grid for E=5, K=2 with
    x = 0: the picks must be the first two of the experts sorted by (-key, id)."""
    E, K, H = 5, 2, 8
    x = torch.zeros(1, H, dtype=torch.bfloat16)
    wr = torch.zeros(E, H, dtype=torch.bfloat16)
    levels = [-0.5, 0.0, 0.25, 1.0]
    for code in range(len(levels) ** E):
        b = [levels[(code // len(levels) ** i) % len(levels)] for i in range(E)]
        ids, _, _ = oracle.route(x, wr, _bf16(b), 1, H, E, K)
        want = sorted(range(E), key=lambda e: (-b[e], e))[:K]
        assert ids[0].tolist() == want, (b, ids)


@pytest.mark.parametrize("K", [1, 6, 8, 16])
def test_selection_matches_a_sort_of_torch_fp64_keys(K):
    """Random rows: the logits from a torch fp64 matmul, the keys and a full
    stable sort (a different selection algorithm) agree with the oracle's K
    passes of arg-max."""
    g = torch.Generator().manual_seed(K)
    T, H, E = 5, 96, 32
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    wr = (torch.randn(E, H, generator=g) * 0.2).to(torch.bfloat16)
    bias = (torch.randn(E, generator=g) * 0.05).to(torch.bfloat16)
    ids, w, keys = oracle.route(x, wr, bias, T, H, E, K, scale=1.5)
    logits = x.double() @ wr.double().T
    s = torch.sigmoid(logits)
    k = s + bias.double()
    assert np.allclose(keys, k.numpy(), rtol=0, atol=1e-12)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(k[t, e]), e))[:K]
        assert ids[t].tolist() == order
        sel = s[t, order]
        assert np.allclose(w[t], (1.5 * sel / sel.sum()).numpy(), rtol=1e-12, atol=0)


def test_selected_keys_dominate_the_rest_and_permuting_experts_permutes_picks():
    g = torch.Generator().manual_seed(7)
    T, H, E, K = 4, 64, 20, 6
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    wr = (torch.randn(E, H, generator=g) * 0.3).to(torch.bfloat16)
    bias = (torch.randn(E, generator=g) * 0.1).to(torch.bfloat16)
    ids, w, keys = oracle.route(x, wr, bias, T, H, E, K)
    for t in range(T):
        rest = np.setdiff1d(np.arange(E), ids[t])
        assert keys[t, ids[t]].min() >= keys[t, rest].max()
        assert np.all(np.diff(keys[t, ids[t]]) <= 0)
    perm = torch.randperm(E, generator=g)
    inv = torch.argsort(perm)
    ids2, w2, _ = oracle.route(x, wr[perm], bias[perm], T, H, E, K)
    assert np.array_equal(inv.numpy()[ids], ids2)
    assert np.array_equal(w, w2)


def test_dominant_logit_is_picked_first():
    H, E, K = 16, 9, 3
    x = torch.zeros(1, H)
    x[0, 3] = 4.0
    wr = torch.zeros(E, H)
    wr[7, 3] = 5.0   # logit 20: sigmoid ~ 1
    wr[2, 3] = -5.0  # logit -20: sigmoid ~ 0
    ids, w, _ = oracle.route(x.to(torch.bfloat16), wr.to(torch.bfloat16), None, 1, H, E, K)
    assert ids[0, 0] == 7 and 2 not in ids[0]
    assert ids[0, 1:].tolist() == [0, 1]  # the rest tie at 1/2: lowest indices
