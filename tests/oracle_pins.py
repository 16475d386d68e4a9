"""Pins of the fp64 oracle to things other than itself.

Each ``pin_*`` takes an :class:`oracle.Oracle` and raises ``AssertionError``
when the oracle disagrees with a closed form, a hand-worked golden file, a
brute-force loop, a numpy textbook attention or an invariant.  The tests run
them on the real oracle (all must pass) and on deliberately broken copies of
its C source (at least one must fail for each), so that a dropped term, a
wrong sign, index or transposed operand in the oracle cannot go unnoticed.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from pa_testutil import (caches_from_tokens, read_golden, random_case, textbook_decode,
                         token_views)

FP16, BF16 = 0, 1
TORCH_DT = {FP16: torch.float16, BF16: torch.bfloat16}


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = float(np.max(np.abs(a - b) / (1.0 + np.abs(b)))) if a.size else 0.0
    assert err <= tol, f"{what}: max scaled error {err:.3e} > {tol:.1e}"


def pin_textbook_gqa(orc):
    """Special case = textbook: the oracle equals numpy softmax(scale q K^T) V
    (GQA groups, random physical placement, ragged lengths), both dtypes."""
    for dt in (FP16, BF16):
        q, kc, vc, bt, lens = random_case(11 + dt, S=3, H=4, KH=2, D=16, BS=4, lens=[1, 7, 13],
                                          dtype=TORCH_DT[dt])
        ref = textbook_decode(q, kc, vc, bt, lens, 0.3)
        got = orc.decode(q, kc, vc, bt, lens, 0.3, dt)
        _close(got, ref, 1e-12, "textbook")
    # Head size 80 (ten 8-element key chunks) in 8- and 64-token blocks.
    for BS in (8, 64):
        q, kc, vc, bt, lens = random_case(17 + BS, S=2, H=4, KH=1, D=80, BS=BS, lens=[9, 130],
                                          dtype=torch.bfloat16)
        _close(orc.decode(q, kc, vc, bt, lens, 0.1, BF16), textbook_decode(q, kc, vc, bt, lens, 0.1),
               1e-12, f"textbook D=80 BS={BS}")


def pin_bruteforce_tiny(orc):
    """Brute force with pure-Python loops and flat offsets computed from the
    caches' shapes (np.ravel_multi_index), math.exp softmax."""
    for KH in (1, 2):
        S, H, D, BS = 2, 2, 8, 2
        q, kc, vc, bt, lens = random_case(5 + KH, S=S, H=H, KH=KH, D=D, BS=BS, lens=[5, 3])
        qf = q.to(torch.float64).numpy().ravel()
        kf = kc.to(torch.float64).numpy().ravel()
        vf = vc.to(torch.float64).numpy().ravel()
        scale = float(np.float32(0.7))
        ref = np.zeros((S, H, D))
        for s in range(S):
            for h in range(H):
                kh = h // (H // KH)
                z = []
                for t in range(int(lens[s])):
                    b = int(bt[s, t // BS])
                    acc = 0.0
                    for d in range(D):
                        ki = np.ravel_multi_index((b, kh, d // 8, t % BS, d % 8), kc.shape)
                        acc += qf[np.ravel_multi_index((s, h, d), q.shape)] * kf[ki]
                    z.append(scale * acc)
                mx = max(z)
                e = [math.exp(v - mx) for v in z]
                tot = sum(e)
                for d in range(D):
                    num = 0.0
                    for t in range(int(lens[s])):
                        b = int(bt[s, t // BS])
                        num += e[t] * vf[np.ravel_multi_index((b, kh, d, t % BS), vc.shape)]
                    ref[s, h, d] = num / tot
        got = orc.decode(q, kc, vc, bt, lens, scale, FP16)
        _close(got, ref, 1e-13, "brute force")


def pin_golden_two_token(orc):
    """Hand-worked two-token case (tests/golden/two_token_closed_form.txt)."""
    rows = {r[0]: [float(v) for v in r[1:]] for r in read_golden("two_token_closed_form.txt")}
    D, BS = 8, 16
    for dt in (FP16, BF16):
        tdt = TORCH_DT[dt]
        q = torch.tensor(rows["q"]).view(1, 1, D).to(tdt)
        k_tok = torch.zeros((1, BS, 1, D))
        v_tok = torch.zeros((1, BS, 1, D))
        k_tok[0, 0, 0], k_tok[0, 1, 0] = torch.tensor(rows["k0"]), torch.tensor(rows["k1"])
        v_tok[0, 0, 0], v_tok[0, 1, 0] = torch.tensor(rows["v0"]), torch.tensor(rows["v1"])
        kc, vc = caches_from_tokens(k_tok.to(tdt), v_tok.to(tdt))
        bt = torch.zeros((1, 1), dtype=torch.int32)
        lens = torch.tensor([2], dtype=torch.int32)
        w0, w1 = rows["w"]
        ref = w0 * np.array(rows["v0"]) + w1 * np.array(rows["v1"])
        got = orc.decode(q, kc, vc, bt, lens, rows["scale"][0], dt)
        _close(got[0, 0], ref, 1e-15, "two-token closed form")


def pin_golden_layout(orc):
    """Hand-derived flat offsets (tests/golden/paged_layout_offsets.txt).  A
    bump at one flat offset must show up at exactly the (b, kh, d, o) the
    fixture names: with partition_size 1 every partition is one token, so the
    per-partition max score (K) or partition output (V) locates it."""
    nb, KH, D, BS = 3, 2, 16, 4
    table = [2, 0, 1]                     # logical block j -> physical block table[j]
    L = nb * BS
    bt = torch.tensor([table], dtype=torch.int32)
    lens = torch.tensor([L], dtype=torch.int32)
    scale = 0.25
    for row in read_golden("paged_layout_offsets.txt"):
        cache, b, kh, d, o, off = row[0], *[int(v) for v in row[1:]]
        t_star = table.index(b) * BS + o   # logical token that lives at (b, o)
        kc = torch.zeros((nb, KH, D // 8, BS, 8), dtype=torch.float16)
        vc = torch.zeros((nb, KH, D, BS), dtype=torch.float16)
        q = torch.zeros((1, KH, D), dtype=torch.float16)
        if cache == "key":
            kc.view(-1)[off] = 4.0
            q[0, kh, d] = 1.0
            m, l, o_p = orc.partitions(q, kc, vc, bt, lens, scale, FP16, 1)
            want = np.zeros((KH, L))
            want[kh, t_star] = 4.0 * scale
            _close(m[0], want, 0.0, f"K layout {row}")
        else:
            vc.view(-1)[off] = 4.0
            m, l, o_p = orc.partitions(q, kc, vc, bt, lens, scale, FP16, 1)
            want = np.zeros((KH, L, D))
            want[kh, t_star, d] = 4.0
            _close(o_p[0], want, 0.0, f"V layout {row}")


def pin_seq_len_one(orc):
    """seq_len = 1: the single weight is exactly 1, so out == V of that token, bitwise."""
    q, kc, vc, bt, lens = random_case(21, S=3, H=4, KH=2, D=16, BS=4, lens=[1, 1, 1], MB=3)
    got = orc.decode(q, kc, vc, bt, lens, 0.125, FP16)
    _, v_tok = token_views(kc, vc)
    for s in range(3):
        for h in range(4):
            want = v_tok[int(bt[s, 0]), 0, h // 2].to(torch.float64).numpy()
            assert np.array_equal(got[s, h], want), "seq_len 1 must return V exactly"


def pin_uniform_weights(orc):
    """Identical keys, q = 0 or scale = 0 make every weight 1/L: out = mean of V."""
    q, kc, vc, bt, lens = random_case(31, S=2, H=2, KH=2, D=16, BS=4, lens=[9, 6])
    k_tok, v_tok = token_views(kc, vc)
    k_same = k_tok.clone()
    k_same[:] = k_tok[0, 0]
    kc_same, _ = caches_from_tokens(k_same, v_tok)
    from pa_testutil import gather_sequence
    for variant in ("same_keys", "q_zero", "scale_zero"):
        qq, kk, sc = q, kc, 0.5
        if variant == "same_keys":
            kk = kc_same
        elif variant == "q_zero":
            qq = torch.zeros_like(q)
        else:
            sc = 0.0
        got = orc.decode(qq, kk, vc, bt, lens, sc, FP16)
        for s in range(2):
            _, V = gather_sequence(kc, vc, bt, s, int(lens[s]))
            _close(got[s], V.mean(axis=0), 1e-13, variant)


def pin_shift_invariance(orc):
    """Adding delta to K[.., 0] of every token shifts every score of a query with
    q[0] = 1 by scale*delta; softmax is shift invariant, so out is unchanged.
    (Small-integer K[.., 0] keeps the shifted values exact in fp16.)"""
    q, kc, vc, bt, lens = random_case(41, S=2, H=2, KH=1, D=16, BS=4, lens=[11, 5])
    q[:, :, 0] = 1.0
    k_tok, v_tok = token_views(kc, vc)
    g = torch.Generator().manual_seed(2)
    k1 = k_tok.clone()
    k1[..., 0] = torch.randint(-4, 5, k1[..., 0].shape, generator=g).to(k1.dtype)
    k2 = k1.clone()
    k2[..., 0] = k1[..., 0] + 3
    kc1, vc1 = caches_from_tokens(k1, v_tok)
    kc2, _ = caches_from_tokens(k2, v_tok)
    a = orc.decode(q, kc1, vc1, bt, lens, 0.5, FP16)
    b = orc.decode(q, kc2, vc1, bt, lens, 0.5, FP16)
    _close(a, b, 1e-13, "softmax shift invariance")
    c = orc.decode(q, torch.zeros_like(kc1), vc1, bt, lens, 0.5, FP16)
    assert np.max(np.abs(a - c)) > 1e-3, "output must depend on K"


def pin_permutation_invariance(orc):
    """Moving physical blocks (and rewriting the table) changes nothing, bitwise."""
    q, kc, vc, bt, lens = random_case(51, S=3, H=4, KH=2, D=16, BS=4, lens=[13, 4, 9],
                                      num_blocks=20, MB=4)
    perm = torch.randperm(20, generator=torch.Generator().manual_seed(9))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(20)
    kc2, vc2 = kc[perm].contiguous(), vc[perm].contiguous()  # new block i holds old perm[i]
    bt2 = inv[bt.long()].to(torch.int32)
    a = orc.decode(q, kc, vc, bt, lens, 0.4, FP16)
    b = orc.decode(q, kc2, vc2, bt2, lens, 0.4, FP16)
    assert np.array_equal(a, b), "physical placement must not matter"


def pin_partition_invariance(orc):
    """combine(partitions(P)) equals the unpartitioned result for any P (the
    phase-2 identity), and unused partitions hold the sentinels (-inf, 0)."""
    q, kc, vc, bt, lens = random_case(61, S=3, H=4, KH=2, D=16, BS=4, lens=[37, 1, 16], MB=10)
    ref = orc.decode(q, kc, vc, bt, lens, 0.35, FP16)
    for P in (1, 4, 8, 7, 16, 64):
        m, l, o = orc.partitions(q, kc, vc, bt, lens, 0.35, FP16, P)
        out = orc.combine(m, l, o, lens, P)
        _close(out, ref, 1e-12, f"partition size {P}")
        for s in range(3):
            np_s = -(-int(lens[s]) // P)
            assert np.all(np.isneginf(m[s, :, np_s:])) and np.all(l[s, :, np_s:] == 0.0)
            assert np.all(np.isfinite(m[s, :, :np_s])) and np.all(l[s, :, :np_s] >= 1.0)


def pin_empty_sequence(orc):
    """seq_len = 0 gives zeros (l = 0 -> inverse taken as 0) and all-sentinel partitions."""
    q, kc, vc, bt, lens = random_case(71, S=2, H=2, KH=2, D=8, BS=4, lens=[0, 5], MB=2)
    got = orc.decode(q, kc, vc, bt, lens, 0.5, FP16)
    assert np.all(got[0] == 0.0) and np.any(got[1] != 0.0)
    m, l, o = orc.partitions(q, kc, vc, bt, lens, 0.5, FP16, 4)
    assert np.all(np.isneginf(m[0])) and np.all(l[0] == 0.0)
    assert np.all(orc.combine(m, l, o, lens, 4)[0] == 0.0)


def pin_combine_closed_form(orc):
    """Phase-2 combine on hand-set states: (m, l) = (0, 1) and (-inf, 0) returns
    o_0 exactly; equal maxima and sums give the plain mean of the o_p;
    m = (ln 3, 0), l = (1, 1) weighs o_0 : o_1 as 3 : 1."""
    D = 4
    lens = np.array([2 * 5], dtype=np.int32)  # P = 5 -> two partitions
    o = np.zeros((1, 1, 2, D))
    o[0, 0, 0] = [1.0, -2.0, 0.5, 3.0]
    o[0, 0, 1] = [5.0, 1.0, -1.0, 0.0]
    m = np.array([[[0.0, -np.inf]]])
    l = np.array([[[1.0, 0.0]]])
    assert np.array_equal(orc.combine(m, l, o, lens, 5)[0, 0], o[0, 0, 0])
    m = np.array([[[0.7, 0.7]]])
    l = np.array([[[2.0, 2.0]]])
    _close(orc.combine(m, l, o, lens, 5)[0, 0], (o[0, 0, 0] + o[0, 0, 1]) / 2, 1e-15, "equal states")
    m = np.array([[[math.log(3.0), 0.0]]])
    l = np.array([[[1.0, 1.0]]])
    _close(orc.combine(m, l, o, lens, 5)[0, 0], 0.75 * o[0, 0, 0] + 0.25 * o[0, 0, 1], 1e-15,
           "3:1 weights")


def pin_lse_golden_two_token(orc):
    """Hand-worked log-sum-exp of the two-token case: log(e^0 + e^1) = log(1 + e)
    (tests/golden/two_token_closed_form.txt)."""
    rows = {r[0]: [float(v) for v in r[1:]] for r in read_golden("two_token_closed_form.txt")}
    D, BS = 8, 16
    for dt in (FP16, BF16):
        tdt = TORCH_DT[dt]
        q = torch.tensor(rows["q"]).view(1, 1, D).to(tdt)
        k_tok = torch.zeros((1, BS, 1, D))
        k_tok[0, 0, 0], k_tok[0, 1, 0] = torch.tensor(rows["k0"]), torch.tensor(rows["k1"])
        kc, vc = caches_from_tokens(k_tok.to(tdt), torch.zeros((1, BS, 1, D)).to(tdt))
        got = orc.lse(q, kc, vc, torch.zeros((1, 1), dtype=torch.int32),
                      torch.tensor([2], dtype=torch.int32), rows["scale"][0], dt)
        _close(got[0, 0], rows["lse"][0], 1e-15, "two-token log-sum-exp")


def pin_lse_closed_forms(orc):
    """q = 0 makes every score 0, so lse = log L exactly; a one-token sequence has
    lse = its one score, scale * q . k (small integers: exact); no tokens give -inf."""
    q, kc, vc, bt, lens = random_case(81, S=3, H=4, KH=2, D=16, BS=4, lens=[9, 1, 0], MB=3)
    got = orc.lse(torch.zeros_like(q), kc, vc, bt, lens, 0.5, FP16)
    assert np.array_equal(got[0], np.full(4, math.log(9.0))), "q = 0 must give log L"
    assert np.array_equal(got[1], np.zeros(4)) and np.all(np.isneginf(got[2]))
    g = torch.Generator().manual_seed(3)
    qi = torch.randint(-3, 4, q.shape, generator=g).to(torch.float16)
    k_tok, v_tok = token_views(kc, vc)
    ki = torch.randint(-3, 4, k_tok.shape, generator=g).to(torch.float16)
    kci, _ = caches_from_tokens(ki, v_tok)
    got = orc.lse(qi, kci, vc, bt, lens, 0.25, FP16)
    for h in range(4):
        k0 = ki[int(bt[1, 0]), 0, h // 2].to(torch.float64)
        assert got[1, h] == 0.25 * float(qi[1, h].to(torch.float64) @ k0), "one-token lse"


def pin_lse_library(orc):
    """Special case = library routine: scipy.special.logsumexp of the scores
    scale * K q, K gathered densely by torch indexing (GQA, ragged, both dtypes)."""
    from scipy.special import logsumexp
    from pa_testutil import gather_sequence
    for dt in (FP16, BF16):
        q, kc, vc, bt, lens = random_case(91 + dt, S=3, H=4, KH=2, D=16, BS=4, lens=[1, 7, 13],
                                          dtype=TORCH_DT[dt])
        got = orc.lse(q, kc, vc, bt, lens, 0.3, dt)
        sc = float(np.float32(0.3))
        for s in range(3):
            K, _ = gather_sequence(kc, vc, bt, s, int(lens[s]))
            for h in range(4):
                z = sc * (K[:, h // 2, :] @ q[s, h].to(torch.float64).numpy())
                _close(got[s, h], logsumexp(z), 1e-13, "scipy logsumexp")


def pin_lse_partition_identity(orc):
    """combine_lse(partitions(P)) equals the unpartitioned lse for any P (the
    phase-2 identity), -inf for an empty sequence."""
    q, kc, vc, bt, lens = random_case(101, S=3, H=4, KH=2, D=16, BS=4, lens=[37, 0, 16], MB=10)
    ref = orc.lse(q, kc, vc, bt, lens, 0.35, FP16)
    assert np.all(np.isneginf(ref[1]))
    for P in (1, 4, 7, 16, 64):
        m, l, _ = orc.partitions(q, kc, vc, bt, lens, 0.35, FP16, P)
        got = orc.combine_lse(m, l, lens, P)
        assert np.all(np.isneginf(got[1]))
        _close(got[[0, 2]], ref[[0, 2]], 1e-13, f"partition size {P}")


def _mq_case(seed, S, q_len, H, KH, D, BS, lens, dtype=torch.float16):
    """Random multi-query inputs: query [S, q_len, H, D] and paged caches."""
    q, kc, vc, bt, L = random_case(seed, S=S * q_len, H=H, KH=KH, D=D, BS=BS, lens=list(lens) * q_len,
                                   dtype=dtype)
    return q.view(S, q_len, H, D).contiguous(), kc, vc, bt[:S].contiguous(), L[:S].contiguous()


def pin_mq_textbook_causal(orc):
    """Special case = textbook: numpy softmax(scale q K^T + causal mask) V and
    scipy logsumexp of the masked scores, K/V gathered densely by torch
    indexing; row i of a sequence of L tokens sees positions <= L - q_len + i."""
    from scipy.special import logsumexp
    from pa_testutil import gather_sequence
    q, kc, vc, bt, lens = _mq_case(111, S=2, q_len=3, H=4, KH=2, D=16, BS=4, lens=[5, 11])
    out, lse = orc.decode_mq(q, kc, vc, bt, lens, 0.3, FP16)
    sc = float(np.float32(0.3))
    for s in range(2):
        L = int(lens[s])
        K, V = gather_sequence(kc, vc, bt, s, L)
        for i in range(3):
            n = L - 3 + i + 1
            for h in range(4):
                z = sc * (K[:n, h // 2, :] @ q[s, i, h].to(torch.float64).numpy())
                w = np.exp(z - z.max())
                _close(out[s, i, h], (w / w.sum()) @ V[:n, h // 2, :], 1e-13, "causal textbook")
                _close(lse[s, i, h], logsumexp(z), 1e-13, "causal logsumexp")


def pin_mq_uniform_causal_bounds(orc):
    """q = 0 makes every visible weight equal: row i's output is the plain mean of V
    over positions 0 .. L - q_len + i and its lse is log of that count, exactly
    pinning each row's causal bound (L = q_len leaves row 0 one token)."""
    from pa_testutil import gather_sequence
    q, kc, vc, bt, lens = _mq_case(121, S=2, q_len=4, H=2, KH=1, D=8, BS=4, lens=[4, 10])
    out, lse = orc.decode_mq(torch.zeros_like(q), kc, vc, bt, lens, 0.5, FP16)
    for s in range(2):
        L = int(lens[s])
        _, V = gather_sequence(kc, vc, bt, s, L)
        for i in range(4):
            n = L - 4 + i + 1
            for h in range(2):
                _close(out[s, i, h], V[:n, 0, :].mean(axis=0), 1e-14, f"mean of {n} tokens")
                assert lse[s, i, h] == math.log(n), "lse of n equal scores is log n"
    _, V0 = gather_sequence(kc, vc, bt, 0, 1)
    assert np.array_equal(out[0, 0, 0], V0[0, 0]), "row 0 with L = q_len sees exactly token 0"


def pin_e4m3_library(orc):
    """Special case = library routine: every one of the 256 E4M3 codes decodes
    to torch.float8_e4m3fn's value (NaN exactly where torch gives NaN)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.e4m3_decode(codes.numpy())
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok]) and np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def pin_e4m3_golden(orc):
    """Hand-derived E4M3 values (tests/golden/e4m3_codes.txt)."""
    rows = read_golden("e4m3_codes.txt")
    got = orc.e4m3_decode(np.array([int(r[0], 16) for r in rows], dtype=np.uint8))
    for (code, value, *_), g in zip(rows, got):
        v = float(value)
        assert (math.isnan(g) and math.isnan(v)) or (g == v and math.copysign(1, g) == math.copysign(1, v)), code


def pin_fp8kv_textbook(orc):
    """Special case = textbook: numpy softmax(scale q (k_scale K)^T) (v_scale V)
    with K and V decoded by torch's float8_e4m3fn and gathered through the block
    table from token-major views obtained by permuting the caches' axes."""
    from pa_testutil import fp8_random_case
    for dt in (FP16, BF16):
        q, kc, vc, bt, lens = fp8_random_case(131 + dt, S=3, H=4, KH=2, D=32, BS=4, lens=[1, 7, 13],
                                              qdtype=TORCH_DT[dt])
        out, lse = orc.decode_fp8kv(q, kc, vc, bt, lens, 0.3, 0.5, 2.0, dt)
        nb, KH, dx, BS, x = kc.shape
        k_tok = kc.view(torch.float8_e4m3fn).to(torch.float64).permute(0, 3, 1, 2, 4).reshape(nb, BS, KH, dx * x)
        v_tok = vc.view(torch.float8_e4m3fn).to(torch.float64).permute(0, 3, 1, 2)
        sc = float(np.float32(0.3))
        for s in range(3):
            L = int(lens[s])
            t = torch.arange(L)
            b = bt[s].long()[t // BS]
            K, V = (0.5 * k_tok[b, t % BS]).numpy(), (2.0 * v_tok[b, t % BS]).numpy()
            for h in range(4):
                z = sc * (K[:, h // 2, :] @ q[s, h].to(torch.float64).numpy())
                w = np.exp(z - z.max())
                _close(out[s, h], (w / w.sum()) @ V[:, h // 2, :], 1e-13, "fp8 textbook")
                _close(lse[s, h], z.max() + math.log(w.sum()), 1e-13, "fp8 lse")


def pin_fp8kv_scales(orc):
    """Scales act as multipliers: v_scale 2 doubles the output exactly, and
    k_scale 2 with scale s equals k_scale 1 with scale 2 s exactly."""
    from pa_testutil import fp8_random_case
    q, kc, vc, bt, lens = fp8_random_case(141, S=2, H=2, KH=1, D=32, BS=4, lens=[9, 3])
    a, la = orc.decode_fp8kv(q, kc, vc, bt, lens, 0.25, 1.0, 1.0, FP16)
    b, lb = orc.decode_fp8kv(q, kc, vc, bt, lens, 0.25, 1.0, 2.0, FP16)
    assert np.array_equal(b, 2.0 * a) and np.array_equal(la, lb)
    c, lc = orc.decode_fp8kv(q, kc, vc, bt, lens, 0.25, 2.0, 1.0, FP16)
    d, ld = orc.decode_fp8kv(q, kc, vc, bt, lens, 0.5, 1.0, 1.0, FP16)
    assert np.array_equal(c, d) and np.array_equal(lc, ld)
    assert np.max(np.abs(c - a)) > 1e-6, "k_scale must matter"



def _mq_fp8_case(seed, S, q_len, H, KH, D, BS, lens, qdtype=torch.float16):
    """Random multi-query inputs over E4M3 code caches: query [S, q_len, H, D]."""
    from pa_testutil import fp8_random_case
    q, kc, vc, bt, L = fp8_random_case(seed, S=S * q_len, H=H, KH=KH, D=D, BS=BS, lens=list(lens) * q_len,
                                       qdtype=qdtype)
    return q.view(S, q_len, H, D).contiguous(), kc, vc, bt[:S].contiguous(), L[:S].contiguous()


def pin_mq_fp8kv_textbook(orc):
    """Special case = textbook: numpy softmax(scale q (k_scale K)^T + causal mask)
    (v_scale V) per query row, K and V decoded by torch's float8_e4m3fn from
    token-major views of the caches; row i of L tokens sees positions <= L - q_len + i."""
    for dt in (FP16, BF16):
        q, kc, vc, bt, lens = _mq_fp8_case(171 + dt, S=2, q_len=3, H=4, KH=2, D=32, BS=4, lens=[3, 13],
                                           qdtype=TORCH_DT[dt])
        out, lse = orc.decode_mq_fp8kv(q, kc, vc, bt, lens, 0.3, 0.5, 2.0, dt)
        nb, KH, dx, BS, x = kc.shape
        k_tok = kc.view(torch.float8_e4m3fn).to(torch.float64).permute(0, 3, 1, 2, 4).reshape(nb, BS, KH, dx * x)
        v_tok = vc.view(torch.float8_e4m3fn).to(torch.float64).permute(0, 3, 1, 2)
        sc = float(np.float32(0.3))
        for s in range(2):
            L = int(lens[s])
            t = torch.arange(L)
            b = bt[s].long()[t // BS]
            K, V = (0.5 * k_tok[b, t % BS]).numpy(), (2.0 * v_tok[b, t % BS]).numpy()
            for i in range(3):
                n = L - 3 + i + 1
                for h in range(4):
                    z = sc * (K[:n, h // 2, :] @ q[s, i, h].to(torch.float64).numpy())
                    w = np.exp(z - z.max())
                    _close(out[s, i, h], (w / w.sum()) @ V[:n, h // 2, :], 1e-13, "fp8 causal textbook")
                    _close(lse[s, i, h], z.max() + math.log(w.sum()), 1e-13, "fp8 causal lse")


def pin_mq_fp8kv_reductions(orc):
    """Reductions to pinned functions, bitwise: one query row is decode_fp8kv; with
    unit scales the E4M3 values, exact in fp16, stored in fp16 caches of the x = 8
    layout give decode_mq's result."""
    q, kc, vc, bt, lens = _mq_fp8_case(181, S=3, q_len=1, H=6, KH=3, D=32, BS=8, lens=[1, 9, 30])
    out, lse = orc.decode_mq_fp8kv(q, kc, vc, bt, lens, 0.2, 1.5, 0.75, FP16)
    ref, ref_lse = orc.decode_fp8kv(q[:, 0], kc, vc, bt, lens, 0.2, 1.5, 0.75, FP16)
    assert np.array_equal(out[:, 0], ref) and np.array_equal(lse[:, 0], ref_lse), "q_len 1 is decode_fp8kv"
    q, kc, vc, bt, lens = _mq_fp8_case(191, S=2, q_len=4, H=4, KH=2, D=32, BS=4, lens=[4, 11])
    out, lse = orc.decode_mq_fp8kv(q, kc, vc, bt, lens, 0.3, 1.0, 1.0, FP16)
    nb, KH, dx, BS, x = kc.shape
    k_tok = kc.view(torch.float8_e4m3fn).permute(0, 3, 1, 2, 4).reshape(nb, BS, KH, dx * x).to(torch.float16)
    v_tok = vc.view(torch.float8_e4m3fn).permute(0, 3, 1, 2).to(torch.float16)
    kc16, vc16 = caches_from_tokens(k_tok.contiguous(), v_tok.contiguous())
    ref, ref_lse = orc.decode_mq(q, kc16, vc16, bt, lens, 0.3, FP16)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse), "unit scales are decode_mq on the values"


def pin_fp32_textbook(orc):
    """Special case = textbook: numpy softmax(scale q K^T) V (and max + log sum
    of the scores) on fp32 caches whose token-major views come from permuting
    the axes of the x = 4 layout (GQA, ragged lengths, an empty sequence)."""
    from pa_testutil import f32_random_case
    for KH, G in ((2, 2), (1, 4)):
        q, kc, vc, bt, lens = f32_random_case(151 + G, S=4, H=KH * G, KH=KH, D=24, BS=4, lens=[1, 6, 13, 0])
        out, lse = orc.decode_fp32(q, kc, vc, bt, lens, 0.3)
        _close(out, textbook_decode(q, kc, vc, bt, lens, 0.3), 1e-13, "fp32 textbook")
        k_tok, _ = token_views(kc, vc)
        for s in range(4):
            L = int(lens[s])
            if L == 0:
                assert np.all(out[s] == 0) and np.all(lse[s] == -np.inf)
                continue
            t = torch.arange(L)
            K = k_tok[bt[s].long()[t // 4], t % 4].to(torch.float64).numpy()
            for h in range(KH * G):
                z = float(np.float32(0.3)) * (K[:, h // G, :] @ q[s, h].to(torch.float64).numpy())
                _close(lse[s, h], z.max() + math.log(np.exp(z - z.max()).sum()), 1e-13, "fp32 lse")


def pin_fp32_equals_16bit(orc):
    """Invariant: fp16 values widened to fp32 (exactly) and stored in the x = 4
    layout give the 16-bit oracle's result on the x = 8 layout, bitwise."""
    q, kc, vc, bt, lens = random_case(161, S=3, H=4, KH=2, D=32, BS=4, lens=[5, 11, 2])
    k_tok, v_tok = token_views(kc, vc)
    from pa_testutil import f32_caches_from_tokens
    kc4, vc4 = f32_caches_from_tokens(k_tok.float(), v_tok.float())
    out, lse = orc.decode_fp32(q.float(), kc4, vc4, bt, lens, 0.3)
    assert np.array_equal(out, orc.decode(q, kc, vc, bt, lens, 0.3, FP16))
    assert np.array_equal(lse, orc.lse(q, kc, vc, bt, lens, 0.3, FP16))



def _mq_f32_case(seed, S, q_len, H, KH, D, BS, lens):
    """Random multi-query fp32 inputs: query [S, q_len, H, D], caches in the x = 4 layout."""
    from pa_testutil import f32_random_case
    q, kc, vc, bt, L = f32_random_case(seed, S=S * q_len, H=H, KH=KH, D=D, BS=BS, lens=list(lens) * q_len)
    return q.view(S, q_len, H, D).contiguous(), kc, vc, bt[:S].contiguous(), L[:S].contiguous()


def pin_mq_fp32_textbook(orc):
    """Special case = textbook: numpy softmax(scale q K^T + causal mask) V per
    query row on fp32 caches whose token-major views come from permuting the
    axes of the x = 4 layout; row i of L tokens sees positions <= L - q_len + i."""
    q, kc, vc, bt, lens = _mq_f32_case(201, S=2, q_len=3, H=4, KH=2, D=24, BS=4, lens=[3, 14])
    out, lse = orc.decode_mq_fp32(q, kc, vc, bt, lens, 0.3)
    nb, KH, dx, BS, x = kc.shape
    k_tok = kc.to(torch.float64).permute(0, 3, 1, 2, 4).reshape(nb, BS, KH, dx * x)
    v_tok = vc.to(torch.float64).permute(0, 3, 1, 2)
    sc = float(np.float32(0.3))
    for s in range(2):
        L = int(lens[s])
        t = torch.arange(L)
        b = bt[s].long()[t // BS]
        K, V = k_tok[b, t % BS].numpy(), v_tok[b, t % BS].numpy()
        for i in range(3):
            n = L - 3 + i + 1
            for h in range(4):
                z = sc * (K[:n, h // 2, :] @ q[s, i, h].to(torch.float64).numpy())
                w = np.exp(z - z.max())
                _close(out[s, i, h], (w / w.sum()) @ V[:n, h // 2, :], 1e-13, "fp32 causal textbook")
                _close(lse[s, i, h], z.max() + math.log(w.sum()), 1e-13, "fp32 causal lse")


def pin_mq_fp32_reductions(orc):
    """Reductions to pinned functions, bitwise: one query row is decode_fp32; fp16
    values widened to fp32 (exactly) in the x = 4 layout give decode_mq's result
    on the x = 8 layout."""
    from pa_testutil import f32_caches_from_tokens
    q, kc, vc, bt, lens = _mq_f32_case(211, S=3, q_len=1, H=6, KH=3, D=24, BS=8, lens=[1, 9, 30])
    out, lse = orc.decode_mq_fp32(q, kc, vc, bt, lens, 0.2)
    ref, ref_lse = orc.decode_fp32(q[:, 0], kc, vc, bt, lens, 0.2)
    assert np.array_equal(out[:, 0], ref) and np.array_equal(lse[:, 0], ref_lse), "q_len 1 is decode_fp32"
    q, kc, vc, bt, lens = _mq_case(221, S=2, q_len=4, H=4, KH=2, D=32, BS=4, lens=[4, 11])
    k_tok, v_tok = token_views(kc, vc)
    kc4, vc4 = f32_caches_from_tokens(k_tok.float(), v_tok.float())
    out, lse = orc.decode_mq_fp32(q.float(), kc4, vc4, bt, lens, 0.3)
    ref, ref_lse = orc.decode_mq(q, kc, vc, bt, lens, 0.3, FP16)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse), "fp16 values in fp32 are decode_mq"

def _tiled_online_forward(q, K, V, scale, tile):
    """softmax(scale q K^T) V by the tiled online softmax of the forward kernel
    of the page "flash_attention.metal -- Flash Attention Metal Shaders" (one
    query row, no causal mask): per key tile, the tile's scores raise the
    running maximum m, the running sum l and the accumulator are rescaled by
    e^(m_old - m_new), the tile's weights are added; at the end out = acc / l
    (0 when l = 0) and the log-sum-exp is m + log l.  fp64 numpy."""
    m, l = -math.inf, 0.0
    acc = np.zeros(V.shape[1])
    for t0 in range(0, K.shape[0], tile):
        z = scale * (K[t0:t0 + tile] @ q)
        m_new = max(m, float(z.max()))
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        w = np.exp(z - m_new)
        l = l * alpha + float(w.sum())
        acc = acc * alpha + w @ V[t0:t0 + tile]
        m = m_new
    out = acc / l if l > 0 else np.zeros_like(acc)
    return out, (m + math.log(l) if l > 0 else -math.inf)


def pin_flash_tiled_forward(orc):
    """Special case = a second textbook routine: the tiled online-softmax
    forward (tiles of 1, 5 and 64 keys) on densely gathered K/V equals the
    oracle's output and log-sum-exp (GQA, ragged lengths)."""
    for dt in (FP16, BF16):
        q, kc, vc, bt, lens = random_case(171 + dt, S=3, H=4, KH=2, D=16, BS=4, lens=[1, 9, 70],
                                          dtype=TORCH_DT[dt])
        out = orc.decode(q, kc, vc, bt, lens, 0.3, dt)
        lse = orc.lse(q, kc, vc, bt, lens, 0.3, dt)
        k_tok, v_tok = token_views(kc, vc)
        sc = float(np.float32(0.3))
        for s in range(3):
            L = int(lens[s])
            t = torch.arange(L)
            b = bt[s].long()[t // 4]
            K = k_tok[b, t % 4].to(torch.float64).numpy()
            V = v_tok[b, t % 4].to(torch.float64).numpy()
            for h in range(4):
                for tile in (1, 5, 64):
                    o_ref, lse_ref = _tiled_online_forward(q[s, h].to(torch.float64).numpy(), K[:, h // 2, :],
                                                           V[:, h // 2, :], sc, tile)
                    _close(out[s, h], o_ref, 1e-12, f"tiled forward (tile {tile})")
                    _close(lse[s, h], lse_ref, 1e-12, f"tiled forward lse (tile {tile})")


ALL_PINS = [
    pin_textbook_gqa, pin_flash_tiled_forward, pin_bruteforce_tiny, pin_golden_two_token, pin_golden_layout,
    pin_seq_len_one, pin_uniform_weights, pin_shift_invariance, pin_permutation_invariance,
    pin_partition_invariance, pin_empty_sequence, pin_combine_closed_form,
    pin_lse_golden_two_token, pin_lse_closed_forms, pin_lse_library, pin_lse_partition_identity,
    pin_mq_textbook_causal, pin_mq_uniform_causal_bounds,
    pin_e4m3_library, pin_e4m3_golden, pin_fp8kv_textbook, pin_fp8kv_scales,
    pin_mq_fp8kv_textbook, pin_mq_fp8kv_reductions,
    pin_fp32_textbook, pin_fp32_equals_16bit, pin_mq_fp32_textbook, pin_mq_fp32_reductions,
]
