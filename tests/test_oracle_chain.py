"""The oracle's Markov-conditioned draft chain ("Remote DSpark drafter --
wire and state contract", section 2: each step adds the bias row of the
previous sampled token, the anchor at step 0; section 6.3: margin = top1 -
top2 of (base + Markov) logits).  Pins: without a bias, or with a bias row
that does not depend on the token, the chain is the per-row q build and
draft draw already pinned; a bias that forces the next token makes the
tokens follow that map from the previous *sampled* token; margins in closed
form; a refused row refuses the rest of its chain."""
import numpy as np

from oracle import oracle as O

FLT_MAX = np.float32(3.4028235e38)


def per_row(x, temps, seed, req=None):
    B, depth, V = x.shape
    counts, _, _, st = O.q_build(x.reshape(-1, V), temps, 0)
    tok, sst = O.draft_sample(counts, None, None, 0, B, depth, seed, req)
    return counts, tok.reshape(B, depth), st


def test_chain_without_bias_is_the_per_row_path(oracle):
    rng = np.random.default_rng(1)
    B, depth, V = 3, 5, 300
    x = rng.normal(0, 2, (B, depth, V)).astype(np.float32)
    temps = rng.choice([1.0, 0.7], B * depth).astype(np.float32)
    c, t, s, m = O.q_chain(x, temps, None, np.arange(B), 9)
    c2, t2, s2 = per_row(x, temps, 9)
    assert np.array_equal(c, c2) and np.array_equal(t, t2) and np.all(s == 0)


def test_chain_with_token_independent_bias(oracle):
    rng = np.random.default_rng(2)
    B, depth, V = 2, 4, 200
    x = rng.normal(0, 2, (B, depth, V)).astype(np.float32)
    row = rng.normal(0, 1, V).astype(np.float32)
    bias = np.tile(row, (5, 1))
    c, t, s, m = O.q_chain(x, None, bias, np.array([3, 4]), 11)
    c2, t2, s2 = per_row((x + row).astype(np.float32), None, 11)
    assert np.array_equal(c, c2) and np.array_equal(t, t2)


def test_chain_follows_the_previous_sampled_token(oracle):
    V, depth, B = 64, 5, 8
    f = (np.arange(V) * 7 + 3) % V            # the next token forced by the bias
    bias = np.zeros((V, V), np.float32)
    bias[np.arange(V), f] = 40.0
    x = np.zeros((B, depth, V), np.float32)
    anchors = np.arange(B) * 5 + 1
    c, t, s, m = O.q_chain(x, None, bias, anchors, 13)
    assert np.all(s == 0)
    prev = anchors.copy()
    for j in range(depth):
        assert np.array_equal(t[:, j], f[prev])
        prev = t[:, j]
    assert np.allclose(m, 40.0)


def test_margins_closed_form(oracle):
    V = 6
    x = np.array([[[5, 3, 3, -np.inf, 1, 0],        # 2
                   [4, 4, 1, 0, 0, 0],              # tie at the top: 0
                   [-np.inf] * 5 + [2]]],           # one finite value
                 np.float32)
    c, t, s, m = O.q_chain(x, None, None, np.array([0]), 1)
    assert np.all(s == 0)
    assert m[0, 0] == 2.0 and m[0, 1] == 0.0 and m[0, 2] == FLT_MAX


def test_refusal_propagates(oracle):
    rng = np.random.default_rng(3)
    B, depth, V = 2, 4, 100
    x = rng.normal(0, 1, (B, depth, V)).astype(np.float32)
    x[0, 1, 7] = np.nan
    c, t, s, m = O.q_chain(x, None, None, np.array([0, V]), 5)
    s = s.reshape(B, depth)
    assert s[0, 0] == O.OK and np.all(s[0, 1:] == O.NONFINITE)
    assert np.all(t[0, 1:] == -1) and np.all(m[0, 1:] == 0)
    assert np.all(c.reshape(B, depth, V)[0, 1:] == 0)
    assert np.all(s[1] == O.BAD_DRAFT)               # anchor outside [0, V)
