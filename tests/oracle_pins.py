"""Checks that pin the f64 oracle to facts other than itself.

Each check takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  They are run against the real oracle by ``test_oracle_pins.py``
and against copies of the oracle with planted mistakes by
``test_oracle_mutants.py`` (which runs this file as a script, one process per
planted mistake, so a mistake that crashes is also caught).

What each pin rests on:
  * half decoding: numpy's own float16 -> float64 conversion, all 65536 codes;
  * golden fixtures: closed-form cases derived by hand (tests/golden/*.json);
  * brute force: scipy's softmax over K/V rows gathered with numpy indexing;
  * context 1: the single weight is exactly 1, so the output is the V row;
  * q = 0: every score is 0, so the output is the plain mean of the V rows;
  * sharding: the online-softmax merge identity over any partition;
  * window: a window equals the same sequence truncated to its last W rows;
  * page permutation: relabelling physical pages changes nothing;
  * equal K rows / constant V rows / repeated q rows: closed forms;
  * invalid rows: out-of-range page ids and lengths are flagged and zeroed.
"""
from __future__ import annotations

import glob
import json
import os
import sys

import numpy as np
from scipy.special import softmax

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- inputs

def rand_case(rng, B, Hq, Hkv, D, PS, lens, decoys=3, max_pages=None):
    """Random fp16 q and paged K/V with a scattered page table (numpy only)."""
    need = [(L + PS - 1) // PS for L in lens]
    mp = max_pages or max(need + [1])
    P = sum(need) + decoys
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    k = rng.standard_normal((P, PS, Hkv, D)).astype(np.float16)
    v = rng.standard_normal((P, PS, Hkv, D)).astype(np.float16)
    perm = rng.permutation(P).astype(np.int32)
    table = np.full((B, mp), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    return q, k, v, table, np.asarray(lens, dtype=np.int32)


def gather(pages, table, b, lo, hi, h):
    """Rows [lo, hi) of KV head h of sequence b, by numpy fancy indexing."""
    PS = pages.shape[1]
    pos = np.arange(lo, hi)
    return pages[table[b, pos // PS], pos % PS, h, :].astype(np.float64)


def window_lo(L, window):
    return max(0, L - window) if window > 0 else 0


def brute_force(q, k, v, table, lens, scale, window):
    """softmax(scale * K q) V per (b, hq), hq -> kv head hq // G."""
    B, Hq, D = q.shape
    G = Hq // k.shape[2]
    out = np.zeros((B, Hq, D))
    for b in range(B):
        lo = window_lo(int(lens[b]), window)
        for hq in range(Hq):
            K = gather(k, table, b, lo, int(lens[b]), hq // G)
            V = gather(v, table, b, lo, int(lens[b]), hq // G)
            if K.shape[0] == 0:
                continue
            w = softmax(scale * (K @ q[b, hq].astype(np.float64)))
            out[b, hq] = w @ V
    return out


def rel_err(a, b):
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


# ---------------------------------------------------------------- checks

def check_half_decoder(o):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([o.half_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def check_golden(o):
    files = sorted(glob.glob(os.path.join(HERE, "golden", "*.json")))
    assert files
    for f in files:
        g = json.load(open(f))
        q = np.array(g["q"], dtype=np.float16)
        k = np.array(g["k_pages"], dtype=np.float16)
        v = np.array(g["v_pages"], dtype=np.float16)
        t = np.array(g["page_table"], dtype=np.int32)
        L = np.array(g["seq_lens"], dtype=np.int32)
        exp = np.array(g["expected"], dtype=np.float64)
        got = o.decode_attn(q, k, v, t, L, g["scale"], g["window"], threads=2)
        assert np.allclose(got, exp, rtol=1e-12, atol=1e-12), (f, got, exp)


def check_brute_force(o):
    rng = np.random.default_rng(11)
    for (Hq, Hkv, D, PS, lens, window) in [
        (4, 1, 8, 4, [1, 7, 0, 13], 0),
        (8, 2, 16, 4, [9, 16, 3], 5),
        (8, 8, 8, 2, [5, 6], 0),          # G = 1: plain multi-head attention
        (16, 2, 64, 16, [40, 33], 1000),  # window longer than the sequence
        (8, 1, 32, 8, [29, 2, 64], 17),
    ]:
        q, k, v, t, L = rand_case(rng, len(lens), Hq, Hkv, D, PS, lens)
        scale = 1.0 / np.sqrt(D)
        got = o.decode_attn(q, k, v, t, L, scale, window, threads=3)
        ref = brute_force(q, k, v, t, L, scale, window)
        for b in range(len(lens)):
            for hq in range(Hq):
                assert rel_err(got[b, hq], ref[b, hq]) <= 1e-12, (Hq, Hkv, D, b, hq)


def check_context_one(o):
    rng = np.random.default_rng(12)
    PS, Hkv, D = 4, 2, 8
    lens = [1, PS + 1, 2 * PS + 2, 3 * PS + 3, 5 * PS + 4, 2]
    q, k, v, t, L = rand_case(rng, len(lens), 4, Hkv, D, PS, lens)
    # window 1 attends only the last position: every slot of a page is hit
    got = o.decode_attn(q, k, v, t, L, 0.3, 1, threads=2)
    for b, n in enumerate(lens):
        for hq in range(4):
            row = gather(v, t, b, n - 1, n, hq // 2)[0]
            assert np.array_equal(got[b, hq], row), (b, hq)


def check_q_zero_mean(o):
    rng = np.random.default_rng(13)
    lens = [11, 1, 30]
    q, k, v, t, L = rand_case(rng, 3, 6, 3, 16, 4, lens)
    q[:] = 0
    for window in (0, 7):
        got = o.decode_attn(q, k, v, t, L, 0.7, window, threads=2)
        for b, n in enumerate(lens):
            for hq in range(6):
                mean = gather(v, t, b, window_lo(n, window), n, hq // 2).mean(axis=0)
                assert rel_err(got[b, hq], mean) <= 1e-14, (window, b, hq)


def check_sharding_identity(o):
    rng = np.random.default_rng(14)
    lens = [37, 64]
    q, k, v, t, L = rand_case(rng, 2, 4, 2, 16, 8, lens)
    scale = 0.25
    full = o.decode_attn(q, k, v, t, L, scale, 0)
    for trial in range(6):
        for b, n in enumerate(lens):
            cuts = np.sort(rng.choice(np.arange(1, n), size=trial % 4, replace=False))
            bounds = [0] + list(cuts) + [n]
            if trial == 5:  # include empty shards
                bounds = [0, 0] + list(cuts) + [n, n]
            for hq in range(4):
                parts = [o.partial(q, k, v, t, b, hq, scale, lo, hi)
                         for lo, hi in zip(bounds[:-1], bounds[1:])]
                ms, ls, accs = zip(*parts)
                merged = o.merge(ms, ls, np.stack(accs))
                assert rel_err(merged, full[b, hq]) <= 1e-12, (trial, b, hq)


def check_partial_brute_force(o):
    """A shard partial is (max score, sum of shifted exps, shifted weighted V)."""
    rng = np.random.default_rng(19)
    lens = [45]
    q, k, v, t, L = rand_case(rng, 1, 4, 2, 16, 8, lens)
    scale = 0.6
    for lo, hi in [(0, 45), (3, 17), (40, 45), (8, 9)]:
        for hq in range(4):
            m, l, acc = o.partial(q, k, v, t, 0, hq, scale, lo, hi)
            K = gather(k, t, 0, lo, hi, hq // 2)
            V = gather(v, t, 0, lo, hi, hq // 2)
            s = scale * (K @ q[0, hq].astype(np.float64))
            assert abs(m - s.max()) <= 1e-12 * max(1.0, abs(m))
            w = np.exp(s - s.max())
            assert abs(l - w.sum()) <= 1e-12 * w.sum()
            assert rel_err(acc, w @ V) <= 1e-12
    m, l, acc = o.partial(q, k, v, t, 0, 0, scale, 5, 5)
    assert m == -np.inf and l == 0.0 and not np.any(acc)


def check_window_truncation(o):
    rng = np.random.default_rng(15)
    PS, Hkv, D, Hq = 4, 2, 8, 4
    lens = [23, 9]
    q, k, v, t, L = rand_case(rng, 2, Hq, Hkv, D, PS, lens)
    W = 6
    win = o.decode_attn(q, k, v, t, L, 0.5, W)
    for b, n in enumerate(lens):
        lo = window_lo(n, W)
        # a fresh cache holding only positions [lo, n), in new pages
        rows = n - lo
        npg = (rows + PS - 1) // PS
        k2 = np.zeros((npg, PS, Hkv, D), np.float16)
        v2 = np.zeros((npg, PS, Hkv, D), np.float16)
        for h in range(Hkv):
            kr, vr = gather(k, t, b, lo, n, h), gather(v, t, b, lo, n, h)
            for i in range(rows):
                k2[i // PS, i % PS, h] = kr[i]
                v2[i // PS, i % PS, h] = vr[i]
        t2 = np.arange(npg, dtype=np.int32)[None, :]
        trunc = o.decode_attn(q[b:b + 1], k2, v2, t2, np.array([rows], np.int32), 0.5, 0)
        assert np.array_equal(win[b], trunc[0]), b


def check_page_permutation(o):
    rng = np.random.default_rng(16)
    lens = [30, 17, 5]
    q, k, v, t, L = rand_case(rng, 3, 8, 2, 16, 4, lens, decoys=5)
    base = o.decode_attn(q, k, v, t, L, 0.4, 0)
    P = k.shape[0]
    perm = rng.permutation(P)           # new page i holds old page perm[i]
    inv = np.argsort(perm).astype(np.int32)
    t2 = np.where(t >= 0, inv[np.maximum(t, 0)], -1).astype(np.int32)
    moved = o.decode_attn(q, k[perm], v[perm], t2, L, 0.4, 0)
    assert np.array_equal(base, moved)


def check_closed_forms(o):
    rng = np.random.default_rng(17)
    lens = [19, 8]
    q, k, v, t, L = rand_case(rng, 2, 4, 2, 8, 4, lens)
    # every K row equal -> equal scores -> plain mean of V for any q
    k_eq = np.broadcast_to(k[0:1, 0:1], k.shape).copy()
    got = o.decode_attn(q, k_eq, v, t, L, 0.9, 0)
    for b, n in enumerate(lens):
        for hq in range(4):
            assert rel_err(got[b, hq], gather(v, t, b, 0, n, hq // 2).mean(0)) <= 1e-14
    # every V row the same vector c -> output c
    c = rng.standard_normal(8).astype(np.float16)
    v_c = np.broadcast_to(c, v.shape).copy()
    got = o.decode_attn(q, k, v_c, t, L, 0.9, 0)
    assert np.allclose(got, np.broadcast_to(c.astype(np.float64), got.shape), rtol=1e-14,
                       atol=0)
    # repeated q rows inside a GQA group -> identical output rows
    q2 = q.copy()
    q2[:, 1] = q2[:, 0]
    got = o.decode_attn(q2, k, v, t, L, 0.9, 0)
    assert np.array_equal(got[:, 0], got[:, 1])
    assert not np.array_equal(got[:, 0], got[:, 2])


def check_invalid_rows(o):
    rng = np.random.default_rng(18)
    lens = [9, 0, 6, 5]
    q, k, v, t, L = rand_case(rng, 4, 2, 1, 8, 4, lens, max_pages=3)
    t[2, 1] = k.shape[0]          # page id past the pool, inside the attended range
    L[3] = 3 * 4 + 1              # longer than max_pages * page_size
    out, err = o.decode_attn(q, k, v, t, L, 0.5, 0, return_errors=True)
    err = err.reshape(4, 2)
    assert err[0].tolist() == [0, 0] and err[1].tolist() == [0, 0]
    assert err[2].tolist() == [1, 1] and err[3].tolist() == [1, 1]
    assert np.all(out[1:] == 0)
    assert np.any(out[0] != 0)


def check_kv_append(o):
    """Scatter of the step's rows: equals numpy fancy-index assignment; the
    rows read back through the table are the new rows bit for bit; every
    other slot is untouched; invalid positions write nothing and are flagged."""
    rng = np.random.default_rng(20)
    lens = [13, 5, 16, 1]
    PS, Hkv, D = 4, 3, 8
    q, k, v, t, L = rand_case(rng, 4, 6, Hkv, D, PS, lens, max_pages=5)
    kn = rng.standard_normal((4, Hkv, D)).astype(np.float16)
    vn = rng.standard_normal((4, Hkv, D)).astype(np.float16)
    pos = np.array([13, -1, 15, 0], dtype=np.int32)   # b=2 overwrites its last slot
    k2, v2, err = o.kv_append(kn, vn, pos, t, k, v)
    ref_k, ref_v = k.copy(), v.copy()
    for b in range(4):
        if pos[b] < 0:
            continue
        ref_k[t[b, pos[b] // PS], pos[b] % PS] = kn[b]
        ref_v[t[b, pos[b] // PS], pos[b] % PS] = vn[b]
    assert np.array_equal(k2, ref_k.view(np.uint16)) and np.array_equal(v2, ref_v.view(np.uint16))
    assert err.tolist() == [0, 0, 0, 0]
    for b in (0, 2, 3):
        for h in range(Hkv):
            got = gather(k2.view(np.float16), t, b, pos[b], pos[b] + 1, h)[0]
            assert np.array_equal(got, kn[b, h].astype(np.float64))
    changed = np.any(k2 != k.view(np.uint16), axis=(2, 3))
    assert changed.sum() <= 3  # at most one (page, slot) per sequence with a row
    # b=1: page id past the pool; b=2: position past its table row (the next
    # row's first entry, b=3's valid page, must not be written through)
    bad_pos = np.array([2, 2, 5 * PS, -3], dtype=np.int32)
    t_bad = t.copy()
    t_bad[1, 0] = k.shape[0] + 2
    k3, v3, err = o.kv_append(kn, vn, bad_pos, t_bad, k, v)
    assert err.tolist() == [0, 1, 1, 0]
    written = np.any(k3 != k.view(np.uint16), axis=(2, 3))
    assert written.sum() == 1 and written[t[0, 0], 2]  # only b=0 wrote


def check_multi_query(o):
    """T new query positions per sequence: scipy brute force with an explicit
    causal mask (query t at position L - T + t sees positions up to itself,
    the window counted from there); each query equals the single-query
    definition on the sequence cut after its own position; queries before the
    first cached position give zero rows."""
    rng = np.random.default_rng(21)
    lens = [9, 2, 17]
    T, Hq, Hkv, D, PS = 3, 4, 2, 8, 4
    _, k, v, t, L = rand_case(rng, 3, Hq, Hkv, D, PS, lens)
    q = rng.standard_normal((3, T, Hq, D)).astype(np.float16)
    for window in (0, 4):
        got = o.decode_attn_multi(q, k, v, t, L, 0.45, window)
        for b, n in enumerate(lens):
            for tq in range(T):
                P = n - T + tq
                for hq in range(Hq):
                    if P < 0:
                        assert not np.any(got[b, tq, hq])
                        continue
                    lo = max(0, P + 1 - window) if window > 0 else 0
                    K = gather(k, t, b, lo, P + 1, hq // 2)
                    V = gather(v, t, b, lo, P + 1, hq // 2)
                    w = softmax(0.45 * (K @ q[b, tq, hq].astype(np.float64)))
                    assert rel_err(got[b, tq, hq], w @ V) <= 1e-12, (window, b, tq, hq)
            for tq in range(T):
                cut = np.array([max(0, n - T + tq + 1)], dtype=np.int32)
                single = o.decode_attn(q[b:b + 1, tq], k, v, t[b:b + 1], cut, 0.45, window)
                assert np.array_equal(got[b, tq], single[0])
    one = o.decode_attn_multi(q[:, :1], k, v, t, L - (T - 1), 0.45, 0)
    assert np.array_equal(one[:, 0], o.decode_attn(q[:, 0], k, v, t, L - (T - 1), 0.45, 0))


def bf16_bits_to_f64(bits):
    """bfloat16 is the upper half of an IEEE binary32: decode through numpy's
    float32."""
    with np.errstate(invalid="ignore"):  # NaN codes stay NaN
        return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def check_bf16(o):
    """bfloat16 elements: the decoder on all 65536 codes, then scipy brute
    force on bf16 q/K/V, and a one-position context returns the V row."""
    import oracle
    codes = np.arange(65536, dtype=np.uint32)
    ref = bf16_bits_to_f64(codes)
    got = np.array([o.bf16_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], ref[~nan])
    rng = np.random.default_rng(22)
    lens = [19, 1, 40]
    qf, kf, vf, t, L = rand_case(rng, 3, 8, 2, 16, 8, lens)
    to_bits = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    qb, kb, vb = to_bits(qf), to_bits(kf), to_bits(vf)
    got = o.decode_attn(oracle.as_bf16_bits(qb), oracle.as_bf16_bits(kb),
                        oracle.as_bf16_bits(vb), t, L, 0.3, 0)
    qd, kd, vd = bf16_bits_to_f64(qb), bf16_bits_to_f64(kb), bf16_bits_to_f64(vb)
    for b, n in enumerate(lens):
        for hq in range(8):
            K, V = gather(kd, t, b, 0, n, hq // 4), gather(vd, t, b, 0, n, hq // 4)
            w = softmax(0.3 * (K @ qd[b, hq]))
            assert rel_err(got[b, hq], w @ V) <= 1e-12
    for hq in range(8):  # lens[1] == 1
        assert np.array_equal(got[1, hq], gather(vd, t, 1, 0, 1, hq // 4)[0])


ALL = [check_half_decoder, check_golden, check_brute_force, check_context_one,
       check_q_zero_mean, check_sharding_identity, check_partial_brute_force, check_window_truncation,
       check_page_permutation, check_closed_forms, check_invalid_rows, check_kv_append,
       check_multi_query, check_bf16]


def run_all(o):
    """Returns the names of the checks that failed."""
    failed = []
    for chk in ALL:
        try:
            chk(o)
        except AssertionError:
            failed.append(chk.__name__)
    return failed


if __name__ == "__main__":  # python tests/oracle_pins.py <variant.so>: exit 1 if any pin fails
    sys.path.insert(0, os.path.dirname(HERE))
    import ctypes
    import oracle
    o = oracle.Oracle(oracle._bind(ctypes.CDLL(sys.argv[1])))
    bad = run_all(o)
    print("FAILED:" + ",".join(bad) if bad else "ALL PASS")
    sys.exit(1 if bad else 0)
