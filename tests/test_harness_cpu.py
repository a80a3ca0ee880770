"""The GPU-parity comparison helpers catch planted mistakes (planted in the
oracle's results, on the CPU): a flipped h code away from a rounding boundary,
a swapped expert pick, an off-by-one permutation."""
import numpy as np
import pytest

import synth
from tests import helpers as Hp


@pytest.fixture(scope="module")
def orc():
    cfg = synth.get_config("mid_ragged")
    w = Hp.layer_weights(cfg)
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed)
    return cfg, Hp.run_oracle(cfg, x, w)


def test_identical_results_pass(orc):
    cfg, o = orc
    pairs = Hp.perm_pairs(o["perm"], cfg.top_k)
    assert Hp.compare_h(cfg, o["hq"], o["hs"], o, pairs) == 0
    gpu = dict(logits=o["logits"].astype(np.float32), idx=o["idx"], weights=o["w"].astype(np.float32))
    assert Hp.compare_routing(cfg, gpu, o) >= 0


def test_planted_h_code_flip_is_caught(orc):
    cfg, o = orc
    pairs = Hp.perm_pairs(o["perm"], cfg.top_k)
    flags = Hp.h_flip_candidates(o, pairs, cfg.h_tensor_scale)
    r, c = np.argwhere(~flags)[len(np.argwhere(~flags)) // 2]
    bad = o["hq"].copy()
    bad[r, c // 2] ^= 0x1 << (4 * (c % 2))     # change one code by one step
    with pytest.raises(AssertionError):
        Hp.compare_h(cfg, bad, o["hs"], o, pairs)


def test_planted_scale_change_is_caught(orc):
    cfg, o = orc
    pairs = Hp.perm_pairs(o["perm"], cfg.top_k)
    bad = o["hs"].copy()
    bad[3, 1] += 1
    with pytest.raises(AssertionError):
        Hp.compare_h(cfg, o["hq"], bad, o, pairs)


def test_planted_routing_mistake_is_caught(orc):
    cfg, o = orc
    idx = o["idx"].copy()
    t = int(np.nonzero(~__import__("oracle").router.near_tie_tokens(o["logits"], cfg.top_k,
                                                                        Hp.TAU))[0][0])
    idx[t, [0, 1]] = idx[t, [1, 0]]
    gpu = dict(logits=o["logits"].astype(np.float32), idx=idx, weights=o["w"].astype(np.float32))
    with pytest.raises(AssertionError):
        Hp.compare_routing(cfg, gpu, o)


def test_logit_error_is_caught(orc):
    cfg, o = orc
    lg = o["logits"].astype(np.float32).copy()
    lg[0, 0] += 1e-3
    gpu = dict(logits=lg, idx=o["idx"], weights=o["w"].astype(np.float32))
    with pytest.raises(AssertionError):
        Hp.compare_routing(cfg, gpu, o)


def test_sign_of_zero_code_is_open_only_near_zero(orc):
    cfg, o = orc
    pairs = Hp.perm_pairs(o["perm"], cfg.top_k)
    flags = Hp.h_flip_candidates(o, pairs, cfg.h_tensor_scale)
    codes = __import__("oracle").quant.unpack_codes(o["hq"])
    # a zero-magnitude code whose h is far from 0 relative to its bound is not open
    zero_far = (codes & 7) == 0
    assert (~flags & zero_far).any()


def test_weight_tolerance_covers_logit_perturbations(orc):
    """weight_tol(w, e) bounds the change of the renormalised softmax weights
    under any logit change of at most e (checked on random and worst-sign
    perturbations of the oracle's selected logits)."""
    import oracle.router as OR
    cfg, o = orc
    rng = np.random.default_rng(5)
    sel = np.take_along_axis(o["logits"], o["idx"], axis=1)
    w0 = OR.renormalised_softmax(sel)
    for e in (1e-6, 1e-5, Hp.LOGIT_TOL):
        for d in (rng.uniform(-e, e, sel.shape),
                  np.where(np.arange(sel.shape[1]) == 0, e, -e) * np.ones_like(sel)):
            w1 = OR.renormalised_softmax(sel + d)
            assert np.all(np.abs(w1 - w0) <= Hp.weight_tol(w0, e) - 1e-6 + 1e-15)


def test_weight_error_beyond_tolerance_is_caught(orc):
    cfg, o = orc
    w = o["w"].astype(np.float32).copy()
    t = int(np.nonzero(~__import__("oracle").router.near_tie_tokens(o["logits"], cfg.top_k,
                                                                        Hp.TAU))[0][0])
    w[t, 0] += 3e-6                        # logits exact: only the 1e-6 fp32 allowance is open
    gpu = dict(logits=o["logits"].astype(np.float32), idx=o["idx"], weights=w)
    with pytest.raises(AssertionError):
        Hp.compare_routing(cfg, gpu, o)
