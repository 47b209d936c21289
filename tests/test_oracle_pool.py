"""The process pool the full-size parity tests use (CPU only): its per-head
error sums equal a direct comparison, and a planted error in one element of
one head is found."""
import math

import numpy as np

import oracle
from sdpa_inputs import make_random
from tests.oracle_pool import backward_head, forward_head, make_pool


def test_pool_error_sums_equal_a_direct_comparison():
    B, H, N, d = 1, 3, 70, 16
    q, k, v, do = (make_random((B, H, N, d), 900 + i) for i in range(4))
    s = 1 / math.sqrt(d)
    O, lse = oracle.attention_forward(q, k, v, s, True)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, s, True)
    O = O.astype(np.float32)
    O[0, 2, 33, 5] += 0.25  # planted error: one element of one head
    tasks = [(q[0, h], k[0, h], v[0, h], do[0, h], O[0, h], lse[0, h], dq[0, h], dk[0, h], dv[0, h], s, True, h)
             for h in range(H)]
    pool, n = make_pool(1 << 20)
    assert n >= 1
    with pool:
        parts = pool.map(backward_head, tasks)
        fparts = pool.map(forward_head, [t[:3] + t[4:6] + (s, True, 0, d, t[-1]) for t in tasks])
    assert [p["o_max"] > 0.2 for p in parts] == [False, False, True]
    assert abs(max(p["o_max"] for p in parts) - 0.25) < 1e-6
    assert parts[2]["o_max_at"][:2] == (33, 5) and parts[2]["head"] == 2
    direct = np.abs(O.astype(np.float64) - oracle.attention_forward(q, k, v, s, True)[0])
    assert abs(sum(p["o_sum"] for p in parts) - direct.sum()) < 1e-9
    assert sum(p["o_n"] for p in parts) == direct.size
    for p, fp in zip(parts, fparts):
        assert p["o_max"] == fp["o_max"] and p["pad_zero"]
        for g in ("dq", "dk", "dv"):
            assert p[g + "_head"] < 1e-6  # float32 rounding of the oracle's own values


def test_workers_report_zero_error_on_the_oracles_own_outputs():
    # Each worker of the full-size tests, fed the oracle's own results as the
    # outputs under test, reports no error; a planted error is found.
    from sdpa_inputs import distance_bias, prefix_lm_mask, e4m3_decode, quantize_e4m3
    from tests.oracle_pool import cross_head, fp8_head, masked_head, window_head
    s = 0.25
    q, k, v, do = (make_random((1, 1, n, 16), 950 + i)[0, 0] for i, n in enumerate((40, 70, 70, 40)))
    one = lambda a: a[None, None]
    O, lse = oracle.attention_forward(one(q), one(k), one(v), s, True, q_offset=30)
    g = oracle.attention_backward(one(q), one(k), one(v), one(do), s, True, q_offset=30)
    p = cross_head((q, k, v, do, O[0, 0], lse[0, 0], g[0][0, 0], g[1][0, 0], g[2][0, 0], s, True, "x"))
    assert p["o_max"] < 1e-12 and p["lse_max"] < 1e-12 and p["dq_head"] < 1e-12 and p["dead_ok"]
    O2 = O[0, 0].copy()
    O2[5, 3] += 0.5
    assert abs(cross_head((q, k, v, None, O2, lse[0, 0], None, None, None, s, True, "x"))["o_max"] - 0.5) < 1e-9
    q, k, v, do = (make_random((1, 1, 90, 16), 960 + i)[0, 0] for i in range(4))
    for recipe, mask, bias in ((("prefix", 20), prefix_lm_mask(90, 20), None),
                               (("distance", 0.1), None, distance_bias(90, 0.1))):
        O, lse = oracle.attention_masked_forward(one(q), one(k), one(v), s, False, None, None, mask, bias)
        g = oracle.attention_masked_backward(one(q), one(k), one(v), one(do), s, False, None, None, mask, bias)
        p = masked_head((q, k, v, do, O[0, 0], lse[0, 0], g[0][0, 0], g[1][0, 0], g[2][0, 0], s, False, recipe, 1))
        assert p["o_max"] < 1e-12 and p["dv_head"] < 1e-12
    q, k, v = (make_random((1, 1, 300, 16), 970 + i)[0, 0] for i in range(3))
    O, lse = oracle.attention_masked_forward(one(q), one(k), one(v), s, True, (50, -1))
    p = window_head((q, k, v, O[0, 0], lse[0, 0], s, 50, 2))
    assert p["o_max"] < 1e-12 and p["lse_max"] < 1e-12
    qd, kd, vd = (e4m3_decode(b) * sc for b, sc in (quantize_e4m3(make_random((200, 32), 980 + i)) for i in range(3)))
    O, lse = oracle.attention_forward(one(qd), one(kd), one(vd), s, True)
    p = fp8_head((qd, kd, vd, O[0, 0], lse[0, 0], s, True, 0, 3))
    assert p["rel_fro"] < 1e-12 and 1e-4 < p["rel_fro_model"] < 0.1
