"""The synthetic inputs follow the stated recipe (no GPU): outlier channels and log-normal norms for
the main-layout workloads, a 2% Student-t(3) mix for the alternate ones, N(0, 1) queries, uniform
ragged lengths and permuted block tables."""
import numpy as np
from scipy import stats

import synth


def test_main_kv_outlier_channels_and_lognormal_norms():
    d, n_kv, n_tok = 128, 4, 4096
    k, v = synth.kv_main(3, 1, n_kv, n_tok, d)
    assert k.dtype == np.float16 and v.dtype == np.float16 and k.shape == (1, n_kv, n_tok, d)
    for x in (k, v):
        x = x[0].astype(np.float64)
        for h in range(n_kv):
            rms = np.sqrt(np.mean(x[h] ** 2, axis=0))
            order = np.argsort(rms)[::-1]
            # exactly four channels scaled by 10
            assert 8.0 < rms[order[3]] / np.median(rms) < 12.5 and rms[order[4]] / np.median(rms) < 1.3
            # one log-normal factor per token vector: over the d - 4 ordinary channels,
            # ln(|x| / sqrt(d - 4)) ~ N(0, 0.5^2) plus chi noise of sd 1/sqrt(2 (d - 4))
            normal = np.sort(order[4:])
            ln = np.log(np.linalg.norm(x[h][:, normal], axis=-1) / np.sqrt(d - 4))
            assert abs(ln.mean()) < 0.03 and 0.47 < ln.std() < 0.54
    # K and V draw their outlier channels separately
    kk = np.argsort(np.sqrt(np.mean(k[0, 0].astype(np.float64) ** 2, axis=0)))[-4:]
    vv = np.argsort(np.sqrt(np.mean(v[0, 0].astype(np.float64) ** 2, axis=0)))[-4:]
    assert set(kk) != set(vv)


def test_alt_kv_student_t_mix():
    k, v = synth.kv_alt(5, 4, 8, 4096, 64)  # 8.4 M entries each
    for x in (k, v):
        x = x.astype(np.float64).ravel()
        # tail mass beyond 5: 0.02 P(|t_3| > 5) = 3.1e-4; a standard normal gives 5.7e-7
        expect = 0.02 * 2 * stats.t.sf(5.0, 3) + (1 - 0.02) * 2 * stats.norm.sf(5.0)
        got = np.mean(np.abs(x) > 5.0)
        se = np.sqrt(expect * (1 - expect) / x.size)
        assert abs(got - expect) < 5 * se, (got, expect)
        assert abs(np.median(x)) < 0.01


def test_queries_lengths_and_block_tables():
    q = synth.queries(1, 8, 40, 128)
    assert q.dtype == np.float16 and abs(q.astype(np.float64).mean()) < 0.02
    assert abs(q.astype(np.float64).std() - 1.0) < 0.02
    lens = synth.ragged_lengths(7, 4000, 1024, 131072)
    assert lens.min() >= 1024 and lens.max() <= 131072
    assert stats.kstest(lens, stats.randint(1024, 131073).cdf).pvalue > 1e-3
    bt = synth.block_table(7, 16, 64, True)
    assert sorted(bt.ravel().tolist()) == list(range(16 * 64))
    assert not np.array_equal(bt.ravel(), np.arange(16 * 64))
    assert np.array_equal(synth.block_table(7, 2, 8, False).ravel(), np.arange(16))
