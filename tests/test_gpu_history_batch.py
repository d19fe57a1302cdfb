"""fp8_amax_history_update_batch: many delayed-scaling states in one launch end exactly as the
single-state call and the oracle leave them (windows of 1 to 1500, both formats, margins, a NaN
amax flagged in its own record's status only, more records than one launch takes)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import host, require_gpu

pytestmark = pytest.mark.gpu


class _State:
    def __init__(self, L, fmt, margin):
        self.fmt, self.margin = fmt, margin
        self.history = torch.zeros(L, device="cuda")
        self.pos = torch.zeros(1, dtype=torch.int64, device="cuda")
        self.amax = torch.zeros(1, device="cuda")
        self.bias = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.scale = torch.ones(1, device="cuda")
        self.scale_inv = torch.ones(1, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")


def _amaxes(seed, T):
    rng = np.random.default_rng(seed)
    return np.exp2(rng.uniform(-30, 20, T)).astype(np.float32)


def test_batch_matches_single_and_oracle():
    q = require_gpu()
    cfg = [(1, 0, 0), (16, 1, 1), (1024, 0, 0), (1500, 1, 0), (4, 0, 2)]
    T = 7
    batch = [_State(*c) for c in cfg]
    single = [_State(*c) for c in cfg]
    ref = [oracle.HistoryState(L) for L, _, _ in cfg]
    seq = [_amaxes(10 + i, T) for i in range(len(cfg))]
    seq[3][4] = np.nan  # one non-finite amax in record 3, step 4
    for t in range(T):
        for i, (L, fmt, margin) in enumerate(cfg):
            batch[i].amax.fill_(float(seq[i][t]))
            single[i].amax.fill_(float(seq[i][t]))
            ref[i].update(float(seq[i][t]), fmt, margin)
            s = single[i]
            q.fp8_amax_history_update(s.history, s.pos, s.amax, fmt, margin, s.bias, s.scale, s.scale_inv, s.status)
        q.fp8_amax_history_update_batch(batch)
        torch.cuda.synchronize()
        for i in range(len(cfg)):
            b, s, r = batch[i], single[i], ref[i]
            for f in ("history", "pos", "amax", "bias", "scale", "scale_inv", "status"):
                assert np.array_equal(host(getattr(b, f)).view(np.uint8), host(getattr(s, f)).view(np.uint8)), (t, i, f)
            assert host(b.bias)[0] == r.bias[0] and host(b.scale)[0] == r.scale[0] and host(b.pos)[0] == r.pos[0]
            assert host(b.scale_inv)[0] == r.scale_inv[0]
            assert np.array_equal(host(b.history), r.hist, equal_nan=True)
    flags = [int(host(b.status)[0]) for b in batch]
    assert flags[3] & q.STATUS_NONFINITE_AMAX and not any(flags[i] for i in (0, 1, 2, 4))


def test_more_records_than_one_launch():
    q = require_gpu()
    n = 60  # two launches of up to 48 records
    states = [_State(8, i % 2, 0) for i in range(n)]
    vals = _amaxes(99, n)
    for st, v in zip(states, vals):
        st.amax.fill_(float(v))
    q.fp8_amax_history_update_batch(states)
    torch.cuda.synchronize()
    for i, (st, v) in enumerate(zip(states, vals)):
        e, s, si = oracle.scale_triple(float(v), i % 2)
        assert host(st.bias)[0] == e and host(st.scale)[0] == s and host(st.pos)[0] == 1, i
        assert host(st.amax)[0] == 0.0
