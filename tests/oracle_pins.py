"""Pins of the oracle to facts outside itself.

Each pin takes a loaded oracle and raises AssertionError when the oracle disagrees with
what the pages or mathematics fix. None re-types the oracle's own code: decoding uses
the E2M1 field formula of the OCP MX spec (not a table), routing is checked by a full
sort, the permutation by its invariants, the FFN by a dense numpy SwiGLU MLP on
independently decoded weights, and bf16 rounding by a search over neighbouring values.
test_oracle_pins.py runs them on the real oracle and on builds with planted mistakes.
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---- independent decoders --------------------------------------------------------------

def e2m1_from_fields(code: int) -> float:
    """E2M1 from its bit fields: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0."""
    sign = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return -mag if sign else mag


def ue8m0_value(s: int) -> float:
    if s == 0:
        return 0.0
    if s == 255:
        return math.inf
    return math.ldexp(1.0, s - 127)


def decode_mxfp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """[R, K/2] codes + [R, K/32] scales -> float64 [R, K]; element 2i is the low nibble."""
    R = codes.shape[0]
    K = codes.shape[1] * 2
    nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(R, K)
    vals = np.array([e2m1_from_fields(c) for c in range(16)], np.float64)[nib]
    sc = np.array([ue8m0_value(s) for s in range(256)], np.float64)[scales]
    return vals * np.repeat(sc, 32, axis=1)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def dense_swiglu(x: np.ndarray, gu_codes, gu_scales, d_codes, d_scales) -> np.ndarray:
    """y = Wd (silu(Wg x) * (Wu x)) for rows of x (float64 [n, H]) with a dense numpy MLP."""
    Wgu = decode_mxfp4(gu_codes, gu_scales)
    I = Wgu.shape[0] // 2
    g = x @ Wgu[:I].T
    u = x @ Wgu[I:].T
    h = g / (1.0 + np.exp(-g)) * u
    return h @ decode_mxfp4(d_codes, d_scales).T


def nearest_bf16_bits(v: float) -> int:
    """Round-to-nearest-even bf16 by bracketing |v| between consecutive bf16 bit patterns."""
    if v == 0:
        return 0x8000 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    lo, hi = 0, 0x7F80                       # search over non-negative finite patterns
    val = lambda b: float(bf16_to_f64(np.array([b], np.uint16))[0])
    while hi - lo > 1:                       # invariant: val(lo) <= a < val(hi) (hi may be inf)
        mid = (lo + hi) // 2
        if val(mid) <= a:
            lo = mid
        else:
            hi = mid
    dl, dh = a - val(lo), val(hi) - a
    if hi == 0x7F80:                         # between max finite and infinity
        half_ulp_above_max = val(0x7F7F) + (val(0x7F7F) - val(0x7F7E)) / 2
        b = 0x7F80 if a >= half_ulp_above_max else lo   # the tie goes to the even pattern: inf
    elif dl < dh or (dl == dh and lo % 2 == 0):
        b = lo
    else:
        b = hi
    return b | (0x8000 if v < 0 else 0)


# ---- small seeded inputs for the pins (not the workload generator: tiny hand sizes) -----

def _rng(tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(1234 + tag))


def tiny_expert(rng, H, I, lo=118, hi=131):
    return (rng.integers(0, 256, (2 * I, H // 2), dtype=np.uint8),
            rng.integers(lo, hi, (2 * I, H // 32), dtype=np.uint8),
            rng.integers(0, 256, (H, I // 2), dtype=np.uint8),
            rng.integers(lo, hi, (H, I // 32), dtype=np.uint8))


class _Experts:
    def __init__(self, mats):
        self.gate_up_codes, self.gate_up_scales, self.down_codes, self.down_scales = [
            np.ascontiguousarray(np.stack(m)) for m in zip(*mats)]


def random_bf16(rng, shape, scale=1.0):
    from routed_moe_fp4_gb300.synthetic import f32_to_bf16_bits
    return f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


# ---- the pins ---------------------------------------------------------------------------

def pin_e2m1_table(o):
    """OCP MX FP4 fields; doubled values are integers; 16 fp32 entries are 64 bytes."""
    vals = [o.e2m1(c) for c in range(16)]
    for c, v in enumerate(vals):
        ref = e2m1_from_fields(c)
        assert v == ref and math.copysign(1, v) == math.copysign(1, ref), (c, v, ref)
        assert float(2 * v).is_integer()
    assert np.array(vals, np.float32).nbytes == 64
    with open(os.path.join(GOLDEN, "e2m1_table.txt")) as f:
        stored = [float(l.split()[1]) for l in f if l.strip() and not l.startswith("#")]
    assert stored == vals, (stored, vals)


def pin_e8m0(o):
    """UE8M0: 2^(s-127) for 1..254, s=0 -> +0, s=255 -> +inf."""
    for s in range(1, 255):
        assert o.e8m0(s) == math.ldexp(1.0, s - 127), s
    z = o.e8m0(0)
    assert z == 0.0 and math.copysign(1.0, z) > 0
    assert math.isinf(o.e8m0(255)) and o.e8m0(255) > 0


def pin_nibble_order(o):
    """Element 2i is the low nibble of byte i."""
    codes = np.array([[0x21, 0xF7] + [0] * 14], np.uint8)       # K = 32: one scale group
    scales = np.array([[127]], np.uint8)
    got = [o.mxfp4(codes, scales, 32, 0, k) for k in range(4)]
    assert got == [0.5, 1.0, 6.0, -6.0], got
    scales2 = np.array([[125]], np.uint8)
    assert o.mxfp4(codes, scales2, 32, 0, 1) == 0.25


def pin_route_bruteforce(o):
    """Top-k by a full sort on (-key, index) with many exact ties, bias included."""
    rng = _rng(1)
    T, E = 64, 16
    for k in (1, 3, 8):
        s = (rng.integers(0, 9, (T, E)) / 8.0).astype(np.float32)
        b = (rng.integers(-2, 3, E) / 16.0).astype(np.float32)
        idx, w = o.route(s, b, k)
        key = s + b                                         # one fp32 addition per element
        for t in range(T):
            order = sorted(range(E), key=lambda e: (-float(key[t, e]), e))[:k]
            assert list(idx[t]) == order, (k, t, list(idx[t]), order)
    s = rng.random((T, E), dtype=np.float32)
    idx, w = o.route(s, None, 4)
    for t in range(T):
        assert list(idx[t]) == sorted(range(E), key=lambda e: (-float(s[t, e]), e))[:4]


def pin_route_weights(o):
    """Weights sum to 1, equal 1 for k=1, follow the unbiased scores, ignore the bias shift."""
    rng = _rng(2)
    T, E = 40, 32
    s = rng.random((T, E), dtype=np.float32) * 0.9 + 0.05
    b = (rng.standard_normal(E) * 0.3).astype(np.float32)
    for k in (1, 2, 8):
        idx, w = o.route(s, b, k)
        sums = w.astype(np.float64).sum(1)
        assert np.all(np.abs(sums - 1.0) <= k * 2.0 ** -23), (k, sums)
        if k == 1:
            assert np.all(w == 1.0)
        sel = np.take_along_axis(s, idx, 1).astype(np.float64)
        ratio = w.astype(np.float64) / (sel / sel.sum(1, keepdims=True))
        assert np.all(np.abs(ratio - 1.0) < 1e-6), ratio
    idx0, w0 = o.route(s, None, 4)
    idx1, w1 = o.route(s, np.full(E, 0.25, np.float32), 4)
    assert np.array_equal(idx0, idx1)
    assert np.array_equal(w0, w1)


def pin_permute(o):
    """Round trip, counts, exclusive offsets, stable token order inside each group."""
    rng = _rng(3)
    for (T, E, k) in ((37, 9, 3), (5, 4, 4), (1, 8, 2), (64, 256, 8)):
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        cnt, off, src, inv = o.permute(idx, E, with_shared=True)
        assert cnt.sum() == T * k + T and cnt[E] == T
        for e in range(E):
            assert cnt[e] == int((idx == e).sum())
        assert off[0] == 0 and np.all(np.diff(off) == cnt)
        assert len(src) == T * k + T
        rows = inv.reshape(-1)
        assert sorted(rows.tolist()) == list(range(T * k))
        for t in range(T):
            for j in range(k):
                r = inv[t, j]
                assert src[r] == t
                assert off[idx[t, j]] <= r < off[idx[t, j] + 1]
        for g in range(E + 1):
            seg = src[off[g]:off[g + 1]]
            assert np.all(np.diff(seg) > 0), (g, seg)
        assert np.array_equal(src[T * k:], np.arange(T))


def _dense_case(o, with_shared: bool):
    rng = _rng(4 + int(with_shared))
    H, I, I_s, T = 64, 32, 64, 5
    x = random_bf16(rng, (T, H))
    ex = _Experts([tiny_expert(rng, H, I)])
    sh = _Experts([tiny_expert(rng, H, I_s)]) if with_shared else None
    Wr = np.zeros((1, H), np.float32)
    r = o.moe_forward(x, Wr, None, 1, ex, sh)
    xf = bf16_to_f64(x)
    ref = dense_swiglu(xf, ex.gate_up_codes[0], ex.gate_up_scales[0], ex.down_codes[0], ex.down_scales[0])
    if with_shared:
        ref = ref + dense_swiglu(xf, sh.gate_up_codes[0], sh.gate_up_scales[0], sh.down_codes[0],
                                 sh.down_scales[0])
    assert np.all(r["idx"] == 0) and np.all(r["w"] == 1.0)
    err = np.abs(r["out_f64"] - ref).max() / np.abs(ref).max()
    assert err < 1e-12, err


def pin_dense_swiglu(o):
    """E=1, k=1: the layer is a dense SwiGLU MLP (no scaling factor, clamp or extra terms)."""
    _dense_case(o, with_shared=False)
    _dense_case(o, with_shared=True)


def pin_dense_gated(o):
    """Permuted path == all experts on all tokens times the sparse gate matrix, plus shared."""
    rng = _rng(6)
    T, H, E, k, I, I_s = 6, 64, 8, 2, 32, 32
    x = random_bf16(rng, (T, H))
    Wr = (rng.standard_normal((E, H)) * 0.3).astype(np.float32)
    b = (rng.standard_normal(E) * 0.1).astype(np.float32)
    ex = _Experts([tiny_expert(rng, H, I) for _ in range(E)])
    sh = _Experts([tiny_expert(rng, H, I_s)])
    r = o.moe_forward(x, Wr, b, k, ex, sh)
    G = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            G[t, r["idx"][t, j]] += float(r["w"][t, j])
    xf = bf16_to_f64(x)
    ref = dense_swiglu(xf, sh.gate_up_codes[0], sh.gate_up_scales[0], sh.down_codes[0], sh.down_scales[0])
    for e in range(E):
        ye = dense_swiglu(xf, ex.gate_up_codes[e], ex.gate_up_scales[e], ex.down_codes[e], ex.down_scales[e])
        ref = ref + G[:, e:e + 1] * ye
    err = np.abs(r["out_f64"] - ref).max() / np.sqrt((ref ** 2).mean())
    assert err < 1e-12, err
    # the bf16 output is the rounding of the fp64 sum
    for t in range(T):
        for m in range(0, H, 7):
            assert r["out"][t, m] == nearest_bf16_bits(float(r["out_f64"][t, m]))


def pin_tokens_output(o):
    """The token-by-token output for given routing (what the GPU parity checks compare with):
    four experts, top-2 with given weights and the shared expert, against numpy SwiGLUs over
    independently decoded weights combined by the weights."""
    rng = _rng(7)
    T, H, E, k, I, I_s = 5, 64, 4, 2, 64, 32
    x = random_bf16(rng, (T, H))
    ex = _Experts([tiny_expert(rng, H, I) for _ in range(E)])
    sh = _Experts([tiny_expert(rng, H, I_s)])
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    w = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    toks = [4, 0, 2]
    out, out64 = o.tokens_output(x, idx, w, ex, sh, toks)
    xf = bf16_to_f64(x)
    ys = [dense_swiglu(xf, ex.gate_up_codes[e], ex.gate_up_scales[e], ex.down_codes[e], ex.down_scales[e])
          for e in range(E)]
    ref = dense_swiglu(xf, sh.gate_up_codes[0], sh.gate_up_scales[0], sh.down_codes[0], sh.down_scales[0])
    for t in range(T):
        for j in range(k):
            ref[t] = ref[t] + float(w[t, j]) * ys[idx[t, j]][t]
    ref = ref[toks]
    err = np.abs(out64 - ref).max() / np.sqrt((ref ** 2).mean())
    assert err < 1e-12, err
    for n in range(len(toks)):
        for m in range(0, H, 5):
            assert out[n, m] == nearest_bf16_bits(float(out64[n, m]))


def pin_sigmoid(o):
    """sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4, symmetry, increasing in the logit."""
    z = np.array([0.0, math.log(3.0), -math.log(3.0), 2.5, -2.5, 10.0, -10.0, 1e-3, -1e-3])
    s = o.sigmoid(z).astype(np.float64)
    assert s[0] == 0.5
    assert abs(s[1] - 0.75) < 1e-7 and abs(s[2] - 0.25) < 1e-7
    assert np.all(np.abs(s[1::2] + s[2::2] - 1.0) < 1e-7)
    zz = np.linspace(-8, 8, 101)
    ss = o.sigmoid(zz)
    assert np.all(np.diff(ss.astype(np.float64)) >= 0) and ss[-1] > 0.99


def pin_logits(o):
    """fp64 logits equal a numpy matmul of the decoded bf16 x and fp32 router weights."""
    rng = _rng(7)
    T, H, E = 9, 96, 13
    x = random_bf16(rng, (T, H))
    Wr = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    z = o.router_logits(x, Wr)
    ref = bf16_to_f64(x) @ Wr.astype(np.float64).T
    assert np.abs(z - ref).max() <= 1e-12 * np.abs(ref).max(), np.abs(z - ref).max()


def pin_round_bf16(o):
    """Round to nearest even bf16, checked by bracketing: ties, subnormals, overflow."""
    cases = [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -30, -(2.0 + 2.0 ** -7),
             3.0e38, 3.4e38, 1e-39, 2.0 ** -133 * 1.5, 2.0 ** -134, 0.0, -0.0, 123.456, -7.77e-3]
    rng = _rng(8)
    cases += list(rng.standard_normal(300) * 10.0 ** rng.integers(-6, 6, 300))
    for v in cases:
        got = o.round_bf16(float(v))
        ref = nearest_bf16_bits(float(v))
        assert got == ref, (v, hex(got), hex(ref))


# ---- expert residency bank ---------------------------------------------------------------
# The bank keeps routed experts in S device slots. The pins check it against bookkeeping kept
# here from the routing sequence alone: which experts each forward touches, how often each was
# touched and when last; never against the oracle's own state arrays except to read them out.

def bank_routing(rng, E: int, T: int, k: int, hot=None, p_hot: float = 0.0) -> np.ndarray:
    """cnt[E + 1] of one forward: each of T tokens picks k distinct experts (expert `hot` first
    with probability p_hot); cnt[E] = T, the shared expert."""
    cnt = np.zeros(E + 1, np.int32)
    for _ in range(T):
        if hot is not None and rng.random() < p_hot:
            rest = rng.choice([e for e in range(E) if e != hot], k - 1, replace=False)
            picks = [hot] + list(rest)
        else:
            picks = rng.choice(E, k, replace=False)
        for e in picks:
            cnt[e] += 1
    cnt[E] = T
    return cnt


def _bank_bijection(st):
    for e in range(st.E):
        if st.slot_of[e] >= 0:
            assert st.expert_in[st.slot_of[e]] == e, ("slot_of/expert_in disagree", e)
    for s in range(st.S):
        if st.expert_in[s] >= 0:
            assert st.slot_of[st.expert_in[s]] == s, ("expert_in/slot_of disagree", s)


def _bank_run(o, E, S, T, k, forwards, seed, hot=None, p_hot=0.0, check=None):
    """Runs `forwards` seeded forwards through the oracle's bank plan with independent
    bookkeeping (usage counts, last forward that touched each expert)."""
    from oracle.oracle import BankState, bank_plan
    rng = _rng(seed)
    st = BankState(E, S)
    uses = np.zeros(E, np.int64)
    last = np.zeros(E, np.int64)
    for f in range(1, forwards + 1):
        cnt = bank_routing(rng, E, T, k, hot, p_hot)
        touched = [e for e in range(E) if cnt[e] > 0]
        before = st.copy()
        rnd, slot, cop = bank_plan(o, st, cnt, T, k)
        _bank_bijection(st)
        assert int(st.stats[0]) == f
        for e in touched:
            uses[e] += 1
        assert np.array_equal(st.usage.astype(np.int64), uses), "usage is not the count of routed forwards"
        assert int(st.stats[1] - before.stats[1]) + int(st.stats[2] - before.stats[2]) == len(touched)
        assert int(st.stats[2] - before.stats[2]) == int(cop.sum())
        assert all(rnd[e] == -1 and cop[e] == 0 for e in range(E) if cnt[e] == 0)
        if check:
            check(before, st, cnt, touched, rnd, slot, cop, uses, last)
        for e in touched:
            last[e] = f
    return st


def _cache_check(before, st, cnt, touched, rnd, slot, cop, uses, last):
    resident_before = {e for e in range(st.E) if before.slot_of[e] >= 0}
    for e in touched:
        assert st.slot_of[e] >= 0 and slot[e] == st.slot_of[e], ("touched expert not resident", e)
        hit = e in resident_before
        assert rnd[e] == (0 if hit else 1) and cop[e] == (0 if hit else 1), ("round/copy", e)
        if hit:
            assert st.slot_of[e] == before.slot_of[e], ("a resident expert moved", e)
    evicted = [e for e in resident_before if st.slot_of[e] < 0]
    kept = [e for e in resident_before if st.slot_of[e] >= 0 and cnt[e] == 0]
    for v in evicted:
        assert cnt[v] == 0, ("a touched expert was evicted", v)
        # the least used (then least recently used) untouched experts go first
        for u in kept:
            assert (uses[v], last[v]) <= (uses[u], last[u]), ("eviction order", v, u)
    empty = sum(1 for s in range(st.S) if before.expert_in[s] < 0)
    misses = sum(1 for e in touched if e not in resident_before)
    assert len(evicted) == max(0, misses - empty), "evicted while a slot was empty"


def pin_bank_cache(o):
    """Cache forwards (T*k <= S): touched experts become resident, resident ones stay in place,
    and only untouched experts are evicted, least used first."""
    _bank_run(o, E=24, S=10, T=3, k=3, forwards=40, seed=40, check=_cache_check)
    _bank_run(o, E=16, S=6, T=2, k=2, forwards=60, seed=41, hot=5, p_hot=0.7, check=_cache_check)


def pin_bank_full(o):
    """A bank with a slot per expert copies each expert once and never evicts."""
    from oracle.oracle import BankState, bank_plan
    rng = _rng(42)
    E = 12
    st = BankState(E, E)
    seen = set()
    for f in range(30):
        cnt = bank_routing(rng, E, 2, 3)
        bank_plan(o, st, cnt, 2, 3)
        seen |= {e for e in range(E) if cnt[e] > 0}
        assert int(st.stats[2]) == len(seen)
        assert all(st.slot_of[e] >= 0 for e in seen)


def pin_bank_hot_expert(o):
    """An expert routed to by most forwards, once loaded, is never evicted by a rarely used one."""
    from oracle.oracle import BankState, bank_plan
    rng = _rng(43)
    E, S, hot = 20, 4, 7
    st = BankState(E, S)
    for f in range(80):
        cnt = bank_routing(rng, E, 1, 2, hot=hot, p_hot=0.8)
        bank_plan(o, st, cnt, 1, 2)
        if f >= 10:
            assert st.slot_of[hot] >= 0, ("the most used expert was evicted", f)


def _stream_check(before, st, cnt, touched, rnd, slot, cop, uses, last):
    G = st.S // 2
    final = {}
    for q, e in enumerate(touched):
        r = q // G
        assert rnd[e] == r, ("round of the q-th touched expert", e)
        assert slot[e] == (r % 2) * G + q % G, ("slot of the q-th touched expert", e)
        want_copy = not (r < 2 and before.expert_in[slot[e]] == e)
        assert cop[e] == int(want_copy), ("copy decision", e)
        final[int(slot[e])] = e
    for s in range(st.S):
        if s in final:
            assert st.expert_in[s] == final[s], ("last group to use a slot owns it", s)
        elif before.expert_in[s] >= 0 and cnt[before.expert_in[s]] > 0:
            assert st.expert_in[s] == -1, ("a moved expert left a copy behind", s)
        else:
            assert st.expert_in[s] == before.expert_in[s], ("an unused slot changed", s)


def pin_bank_stream(o):
    """Transient forwards (T*k > S): touched experts in increasing order fill alternate halves
    of the bank in groups of S/2; a repeated forward finds its last two groups in place."""
    from oracle.oracle import BankState, bank_plan
    rng = _rng(44)
    E, S = 32, 8
    st = BankState(E, S)
    uses = np.zeros(E, np.int64)
    last = np.zeros(E, np.int64)
    # forward 5 routes 7 tokens x 3 slots to 7 experts (more slots than the bank holds, fewer
    # experts), among them the one in the last slot, which then moves to a lower slot and must
    # leave the last slot empty; forward 6 repeats it
    seq = [(2, 2), (12, 3), (1, 2), (12, 3), (7, 3), (7, 3)]
    few = None
    for f, (T, k) in enumerate(seq, start=1):
        if f == 5:
            pick = {1, 4, 9, 15, 22, 23, 30}
            if st.expert_in[S - 1] >= 0:
                pick = set(sorted(pick - {int(st.expert_in[S - 1])})[:6]) | {int(st.expert_in[S - 1])}
            few = np.zeros(E + 1, np.int32)
            few[sorted(pick)] = 3
            few[E] = 7
        cnt = few if f >= 5 else bank_routing(rng, E, T, k)
        touched = [e for e in range(E) if cnt[e] > 0]
        before = st.copy()
        rnd, slot, cop = bank_plan(o, st, cnt, T, k)
        _bank_bijection(st)
        for e in touched:
            uses[e] += 1
        assert np.array_equal(st.usage.astype(np.int64), uses)
        if min(T * k, E) > S:
            _stream_check(before, st, cnt, touched, rnd, slot, cop, uses, last)
        else:
            _cache_check(before, st, cnt, touched, rnd, slot, cop, uses, last)
        if f == 6:   # the same two groups again: every expert is already in its slot
            assert not cop.any(), "a repeated forward recopied experts in place"
        for e in touched:
            last[e] = f


# ---- FP8 dense projection -----------------------------------------------------------------

def e4m3_values() -> dict:
    """Every finite OCP E4M3 value by construction: normals (1 + m/8) * 2^(e - 7) for exponent
    fields 1..15 (mantissa 7 excluded at 15, that code is NaN), subnormals (m/8) * 2^-6."""
    vals = {}
    for sign in (0, 1):
        for e in range(16):
            for m in range(8):
                if e == 15 and m == 7:
                    continue
                mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
                vals[(sign << 7) | (e << 3) | m] = -mag if sign else mag
    return vals


def pin_e4m3(o):
    """E4M3 against the OCP FP8 spec: 1.0 = 0x38, max 448 = 0x7E, smallest subnormal 2^-9,
    smallest normal 2^-6, NaN at S.1111.111, and every code by its fields."""
    fixed = {0x38: 1.0, 0x7E: 448.0, 0xFE: -448.0, 0x01: 2.0 ** -9, 0x08: 2.0 ** -6, 0x00: 0.0, 0x40: 2.0,
             0x30: 0.5, 0x3C: 1.5, 0x07: 7 * 2.0 ** -9}
    for c, v in fixed.items():
        assert o.e4m3(c) == v, (hex(c), o.e4m3(c), v)
    assert math.isnan(o.e4m3(0x7F)) and math.isnan(o.e4m3(0xFF))
    for c, v in e4m3_values().items():
        assert o.e4m3(c) == v, (hex(c), o.e4m3(c), v)


def fp8_case(rng, T, K, N, pow2_scales=False):
    """x bf16 bits [T, K], E4M3 codes [N, K] (no NaN codes), fp32 block scales."""
    x = random_bf16(rng, (T, K))
    w = rng.integers(0, 256, (N, K), dtype=np.uint8)
    w[(w & 0x7F) == 0x7F] ^= 1                        # NaN codes -> 0x7E / 0xFE
    nb, kb = -(-N // 128), -(-K // 128)
    if pow2_scales:
        sc = (2.0 ** rng.integers(-12, -4, (nb, kb))).astype(np.float32)
    else:
        sc = (rng.uniform(1.0, 2.0, (nb, kb)) * 2.0 ** rng.integers(-12, -4, (nb, kb))).astype(np.float32)
    return x, w, sc


def pin_fp8_linear(o):
    """The projection equals numpy's matmul of the bf16 activations and the weights decoded by
    their E4M3 fields, each 128 x 128 block multiplied by its scale (blocks 2 x 3: a transposed or
    dropped block index fails)."""
    rng = _rng(50)
    table = np.zeros(256)
    for c, v in e4m3_values().items():
        table[c] = v
    for T, K, N in ((3, 384, 256), (1, 128, 128), (5, 256, 384)):
        x, w, sc = fp8_case(rng, T, K, N)
        W = table[w] * np.repeat(np.repeat(sc.astype(np.float64), 128, 0), 128, 1)[:N, :K]
        ref = bf16_to_f64(x) @ W.T
        out, out64 = o.fp8_linear(x, w, sc)
        assert np.allclose(out64, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max()), (T, K, N)
        for v, b in zip(ref.ravel()[:64], out.ravel()[:64]):
            assert b == nearest_bf16_bits(float(v))


# ---- NVFP4 experts ---------------------------------------------------------------------------

def decode_nvfp4(codes: np.ndarray, scales: np.ndarray, glob: float) -> np.ndarray:
    """[R, K] values from E2M1 fields, E4M3 scale fields per 16 along K and the matrix scale."""
    R, K2 = codes.shape
    K = 2 * K2
    e2 = np.array([e2m1_from_fields(c) for c in range(16)])
    e4 = np.zeros(256)
    for c, v in e4m3_values().items():
        e4[c] = v
    lo, hi = codes & 15, codes >> 4
    vals = np.empty((R, K))
    vals[:, 0::2] = e2[lo]
    vals[:, 1::2] = e2[hi]
    return vals * np.repeat(e4[scales], 16, axis=1) * float(glob)


def pin_nvfp4_decode(o):
    """Single weights against the E2M1 and E4M3 field decoders, in both nibbles and across
    16-element groups (a 32-element group or a missing matrix scale fails)."""
    rng = _rng(60)
    R, K = 3, 64
    codes = rng.integers(0, 256, (R, K // 2), dtype=np.uint8)
    scales = rng.integers(0x20, 0x50, (R, K // 16), dtype=np.uint8)
    ref = decode_nvfp4(codes, scales, 0.375)
    for r in range(R):
        for k in range(K):
            assert o.nvfp4(codes, scales, 0.375, K, r, k) == ref[r, k], (r, k)


def pin_nvfp4_dense_swiglu(o):
    """One expert, top-1, no shared expert: the routed layer reduces to a dense SwiGLU MLP over the
    independently decoded NVFP4 weights (numpy), to fp64 rounding."""
    from routed_moe_fp4_gb300 import synthetic as S
    rng = _rng(61)
    H, I, T = 128, 64, 3
    ex = S.make_nv_experts(61, "pin", 1, H, I)
    x = random_bf16(rng, (T, H))
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1), np.float32)
    out, out64 = o.tokens_output_nv(x, idx, w, ex, None, list(range(T)))
    Wgu = decode_nvfp4(ex.gate_up_codes[0], ex.gate_up_scales[0], ex.gate_up_global[0])
    Wd = decode_nvfp4(ex.down_codes[0], ex.down_scales[0], ex.down_global[0])
    xv = bf16_to_f64(x)
    g, u = xv @ Wgu[:I].T, xv @ Wgu[I:].T
    ref = (g / (1.0 + np.exp(-g)) * u) @ Wd.T
    assert np.allclose(out64, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())


def pin_nvfp4_gated(o):
    """Four NVFP4 experts, top-2 with given weights, and the shared expert: each token's output is
    the shared expert's dense SwiGLU plus the weighted SwiGLUs of its two experts, each expert with
    its own codes, scales and matrix scales (numpy over independently decoded weights)."""
    from routed_moe_fp4_gb300 import synthetic as S
    rng = _rng(62)
    H, I, I_s, E, T, k = 64, 32, 64, 4, 5, 2
    ex = S.make_nv_experts(62, "pin-gated", E, H, I)
    sh = S.make_nv_experts(62, "pin-gated-shared", 1, H, I_s)
    # distinct matrix scales per expert, so that taking another expert's scale shows
    ex.gate_up_global[:] = np.float32(2.0) ** np.arange(E, dtype=np.float32) * np.float32(0.75)
    ex.down_global[:] = np.float32(0.5) ** np.arange(E, dtype=np.float32)
    x = random_bf16(rng, (T, H))
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    w = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    out, out64 = o.tokens_output_nv(x, idx, w, ex, sh, list(range(T)))
    xv = bf16_to_f64(x)

    def mlp(e_set, e):
        Wgu = decode_nvfp4(e_set.gate_up_codes[e], e_set.gate_up_scales[e], e_set.gate_up_global[e])
        Wd = decode_nvfp4(e_set.down_codes[e], e_set.down_scales[e], e_set.down_global[e])
        n = Wgu.shape[0] // 2
        g, u = xv @ Wgu[:n].T, xv @ Wgu[n:].T
        return (g / (1.0 + np.exp(-g)) * u) @ Wd.T

    ys = [mlp(ex, e) for e in range(E)]
    ref = mlp(sh, 0)
    for t in range(T):
        for j in range(k):
            ref[t] = ref[t] + float(w[t, j]) * ys[idx[t, j]][t]
    err = np.abs(out64 - ref).max() / np.sqrt((ref ** 2).mean())
    assert err < 1e-12, err


ALL_PINS = [pin_e2m1_table, pin_e8m0, pin_nibble_order, pin_route_bruteforce, pin_route_weights,
            pin_permute, pin_dense_swiglu, pin_dense_gated, pin_tokens_output, pin_sigmoid, pin_logits, pin_round_bf16,
            pin_bank_cache, pin_bank_full, pin_bank_hot_expert, pin_bank_stream, pin_e4m3, pin_fp8_linear,
            pin_nvfp4_decode, pin_nvfp4_dense_swiglu, pin_nvfp4_gated]
