"""Pins of the sampling-chain oracle (oracle/sampling.py) by hand values,
closed forms and the distribution the draw must reproduce."""
import math

import numpy as np

from oracle import sampling as S

OFF = dict(top_p=1.0, min_p=0.0, repeat_penalty=1.0)


def test_temperature_zero_is_argmax_lowest_id_on_ties():
    l = np.array([1.0, 3.0, 3.0, -1.0], np.float32)
    assert S.decide(l, S.Params(temperature=0.0), 0.9)[0] == 1


def test_top_k_one_is_argmax_for_any_u():
    l = np.array([0.1, 2.0, 1.9, -5.0], np.float32)
    for u in (0.0, 0.3, 0.999):
        assert S.decide(l, S.Params(temperature=1.7, top_k=1, **OFF), u)[0] == 1


def test_draw_reproduces_softmax_of_scaled_logits():
    # inverse-CDF sampling over a fine grid of u gives each token its
    # probability softmax(l / T), for a token order given by descending logit
    l = np.array([0.3, -1.2, 2.0, 0.9, 0.0], np.float32)
    T = 0.7
    p = np.exp(l / T - np.max(l / T))
    p /= p.sum()
    n = 20000
    counts = np.zeros(l.size)
    for i in range(n):
        counts[S.decide(l, S.Params(temperature=T, top_k=5, **OFF), (i + 0.5) / n)[0]] += 1
    assert np.allclose(counts / n, p, atol=2e-4)


def test_repeat_penalty_hand_values():
    l = np.array([2.0, -2.0, 1.0, 0.5], np.float32)
    out = S.penalize(l, [0, 1, 0], 2.0, 64)
    assert np.array_equal(out, np.array([1.0, -4.0, 1.0, 0.5], np.float32))
    # only the last n history entries count
    assert np.array_equal(S.penalize(l, [0, 1], 2.0, 1), np.array([2.0, -4.0, 1.0, 0.5], np.float32))


def test_penalty_acts_before_top_k():
    l = np.array([5.0, 4.0, 3.0], np.float32)
    p = S.Params(temperature=1.0, top_k=1, top_p=1.0, min_p=0.0, repeat_penalty=10.0, penalty_last_n=8)
    assert S.decide(l, p, 0.5, history=[0])[0] == 1


def test_top_p_keeps_shortest_prefix_reaching_p_and_renormalizes():
    probs = np.array([0.5, 0.3, 0.2])
    l = np.log(probs).astype(np.float32)
    p = S.Params(temperature=1.0, top_k=3, top_p=0.75, min_p=0.0, repeat_penalty=1.0)
    # kept {0, 1} with mass 0.8: u = 0.6 -> 0.48 < 0.5 -> token 0; u = 0.7 -> 0.56 -> token 1
    assert S.decide(l, p, 0.6)[0] == 0 and S.decide(l, p, 0.7)[0] == 1
    # token 2 is never drawn
    assert all(S.decide(l, p, u)[0] != 2 for u in np.linspace(0, 0.9999, 101))
    # p below the top probability still keeps one token
    assert S.decide(l, S.Params(temperature=1.0, top_k=3, top_p=0.1, min_p=0.0), 0.99)[0] == 0


def test_min_p_threshold_relative_to_top_probability():
    probs = np.array([0.5, 0.3, 0.2])
    l = np.log(probs).astype(np.float32)
    p = S.Params(temperature=1.0, top_k=3, top_p=1.0, min_p=0.5, repeat_penalty=1.0)   # threshold 0.25
    drawn = {S.decide(l, p, u)[0] for u in np.linspace(0, 0.9999, 201)}
    assert drawn == {0, 1}
    # kept mass 0.8: the boundary between tokens 0 and 1 sits at u = 0.5 / 0.8
    assert S.decide(l, p, 0.62)[0] == 0 and S.decide(l, p, 0.63)[0] == 1


def test_top_k_ties_take_lower_id_first():
    l = np.array([1.0, 2.0, 2.0, 2.0, 0.0], np.float32)
    idx, vals = S.top_k(l, 2)
    assert list(idx) == [1, 2] and list(vals) == [2.0, 2.0]


def test_margin_reports_closeness_to_a_boundary():
    probs = np.array([0.5, 0.5])
    l = np.log(probs).astype(np.float32)
    p = S.Params(temperature=1.0, top_k=2, **OFF)
    assert S.decide(l, p, 0.5)[1] < 1e-6          # exactly on the boundary
    assert S.decide(l, p, 0.25)[1] > 0.2
