"""The device-side property checker (tests/_props.py), run on the CPU
against the oracle: it accepts the oracle's selections and rejects planted
mistakes, so a GPU test that relies on it checks something real."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _props


def _case(dtype):
    w = synth.long_decode(seed=77, B=24, H=2, M=300, K=16, dtype=dtype, min_len=1,
                          max_len=300 * 128 + 500)
    nvp = oracle.num_valid_pages_decode(w.seq_lens.numpy(), 1)
    synth.inject_specials(w.scores, seed=78, frac_each=0.02, frac_ties=0.1)
    synth.fill_tail(w.scores, torch.from_numpy(nvp), float("-inf"))
    idx = oracle.topk_select(w.scores, nvp, w.K, w.num_init, w.num_local)
    return w, torch.from_numpy(nvp), torch.from_numpy(idx)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_props_accept_the_oracle(dtype):
    w, nvp, idx = _case(dtype)
    _props.check_selection(w.scores, nvp, idx, w.K, w.num_init, w.num_local)


def _mutations(w, nvp, idx):
    v = torch.clamp(nvp.long(), max=w.M)
    r = int(torch.nonzero(v > 40)[0, 0])
    vr = int(v[r])
    a = idx.clone()
    a[r, 0, 5] = -1                                  # a hole among the used slots
    yield "hole", a
    a = idx.clone()
    a[r, 1, [3, 4]] = a[r, 1, [4, 3]]                # not ascending
    yield "order", a
    a = idx.clone()
    a[r, 0, 0] = 1 if int(a[r, 0, 1]) != 1 else 2    # init block dropped
    a[r, 0] = torch.sort(a[r, 0]).values
    yield "init", a
    a = idx.clone()
    a[r, 0, w.K - 1] = vr                            # id past the causal bound
    yield "bound", a
    # the best unselected block swapped in for the worst selected non-forced one
    keys = _props.order_keys(w.scores[r, 0, :vr])
    chosen = set(int(x) for x in idx[r, 0] if x >= 0)
    forced = {0, vr - 2, vr - 1}
    worst = min((b for b in chosen - forced), key=lambda b: (int(keys[b]), -b))
    best_left = max((b for b in range(vr) if b not in chosen), key=lambda b: (int(keys[b]), -b))
    a = idx.clone()
    row = sorted((chosen - {worst}) | {best_left})
    a[r, 0, :len(row)] = torch.tensor(row, dtype=a.dtype)
    yield "exchange", a


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_props_reject_planted_mistakes(dtype):
    w, nvp, idx = _case(dtype)
    for name, bad in _mutations(w, nvp, idx):
        with pytest.raises(AssertionError):
            _props.check_selection(w.scores, nvp, bad, w.K, w.num_init, w.num_local)
            raise RuntimeError(f"mutation {name} was not caught")
