"""Host checks of the parity protocol's own logic (tests/util.py): the typical-
acceptance outcome enumeration reproduces the oracle's result when no decision
is ambiguous, offers both resolutions of an ambiguous one, and the vectorised
race of the header's random numbers agrees with the oracle's draw."""
import numpy as np

import workloads as W
from oracle import oracle as O
from util import check_typical, race_draw, typical_outcomes


def _case(seed):
    t = O.tree_layout(O.product_tree_paths((3, 3, 2)), 3)
    B, V = 6, 400
    cand = O.build_tree(W.random_topk_lists(seed, B, 3, 3, V), W.root_tokens(seed, B, V), t["depth"], t["rank"])
    logits = W.normal_logits(seed, B, t["N"], V, 1.0)
    for b in range(B):  # make some candidates likely so that paths get long
        for j in range(1, t["N"]):
            if (b + j) % 3:
                logits[b, t["parent"][j], cand[b, j]] += 5.0
    return t, cand, logits


def test_outcomes_without_ambiguity_are_the_oracle_result():
    t, cand, logits = _case(3)
    ref = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"], "typical", 1.0, 0.2, 0.5)
    assert check_typical(ref, ref, t["parent"], t["depth"], band=0.0) == 0
    assert (ref["accept_len"] > 0).any()
    for b in range(len(cand)):
        outs, na = typical_outcomes(ref, b, t["parent"], t["depth"], band=0.0)
        assert na == 0 and len(outs) == 1


def test_an_ambiguous_node_allows_both_decisions_and_nothing_else():
    t, cand, logits = _case(4)
    ref = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"], "typical", 1.0, 0.2, 0.5)
    b = int(np.argmax(ref["accept_len"]))
    best = int(ref["best_node"][b])
    # make the best node's own decision ambiguous: both the result and the one
    # with that node rejected are allowed
    r2 = {k: v.copy() for k, v in ref.items()}
    r2["pcand"][b, best] = r2["tau"][b, t["parent"][best]] * (1 + 1e-7)
    outs, na = typical_outcomes(r2, b, t["parent"], t["depth"], band=1e-6)
    assert na == 1 and len(outs) == 2
    assert (int(ref["accept_len"][b]), best) in {(o[0], o[1]) for o in outs}
    bad = {k: v.copy() for k, v in ref.items()}
    bad["best_node"][b] = 0
    bad["accept_len"][b] = 0
    try:
        check_typical(bad, ref, t["parent"], t["depth"], band=0.0)
        raise RuntimeError("a wrong result passed the check")
    except AssertionError:
        pass


def test_vectorised_race_matches_the_oracle_draw():
    t = O.tree_layout(O.product_tree_paths((2, 2)), 2)
    B, V, T = 4, 3001, 1.0
    cand = O.build_tree(W.random_topk_lists(9, B, 2, 2, V), W.root_tokens(9, B, V), t["depth"], t["rank"])
    logits = W.normal_logits(9, B, t["N"], V, 3.0)
    ref = O.verify_tree_sample(logits, cand, t["parent"], t["depth"], t["max_depth"], 5, 2, T)
    for b in range(B):
        x = logits[b, ref["best_node"][b]].astype(np.float64) / T
        tok, gap = race_draw(np.exp(x - x.max()), O.row_key(5, 4, b, 2, 0))
        assert tok == ref["next_tok"][b]
        assert abs(gap - ref["race_gap"][b]) <= 1e-9 * max(1.0, gap)
