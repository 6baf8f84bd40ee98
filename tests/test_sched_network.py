"""The scheduler's sort network, selection and merge tree, restated on the host (no GPU).

schedule_kernel sorts n_pad = E * threads keys with each thread holding E
consecutive keys in registers: strides below E are exchanged in registers,
strides E .. 32E - 1 between the lanes of a warp, and strides of 32E and more
through shared memory, whose word w sits at w ^ ((w >> 4) & 15). This model
runs the same stages with the same index arithmetic (at fewer threads, which
keeps all three kinds of stage) and checks that the keys come out sorted and
that every lane partner lies in the same warp.

Before any sort, schedule_kernel selects the top survival bins holding at most
1024 candidates (a prefix of the sorted order) and, for B <= 1024, sorts them
with a merge tree over the requests' runs. The models below check that the
selection is exactly the sorted order's first keys, that each request's
selected positions form a prefix, and that the merge tree sorts them.
"""
import random

import pytest


def _swz(w):
    return w ^ ((w >> 4) & 15)


def _cx_shared(mem, i, stride, size):
    lo = 2 * i - (i & (stride - 1))
    hi = lo + stride
    asc = (lo & size) == 0
    a, c = mem[_swz(lo)], mem[_swz(hi)]
    if (a > c) == asc:
        mem[_swz(lo)], mem[_swz(hi)] = c, a


def _sort(keys, threads, E):
    n_pad = threads * E
    mem = [0] * n_pad
    v = [[keys[t * E + j] for j in range(E)] for t in range(threads)]
    size = 2
    while size <= n_pad:
        stride = size >> 1
        if stride >= 32 * E:
            for t in range(threads):
                for j in range(E):
                    mem[_swz(t * E + j)] = v[t][j]
            while stride >= 32 * E:
                for i in range(n_pad // 2):
                    _cx_shared(mem, i, stride, size)
                stride >>= 1
            v = [[mem[_swz(t * E + j)] for j in range(E)] for t in range(threads)]
        while stride >= E:
            d = stride // E
            nv = [[0] * E for _ in range(threads)]
            for t in range(threads):
                assert (t ^ d) // 32 == t // 32, "shuffle partner outside the warp"
                for j in range(E):
                    i = t * E + j
                    o = v[t ^ d][j]
                    keep_min = ((i & stride) == 0) == ((i & size) == 0)
                    nv[t][j] = min(o, v[t][j]) if keep_min else max(o, v[t][j])
            v = nv
            stride >>= 1
        st = E // 2
        while st > 0:
            if st <= stride:
                for t in range(threads):
                    for j in range(E):
                        if (j & st) == 0:
                            asc = ((t * E + j) & size) == 0
                            a, c = v[t][j], v[t][j | st]
                            if (a > c) == asc:
                                v[t][j], v[t][j | st] = c, a
            st >>= 1
        size <<= 1
    return [v[t][j] for t in range(threads) for j in range(E)]


@pytest.mark.parametrize("E", [2, 4, 8])
@pytest.mark.parametrize("ties", [False, True])
def test_register_shuffle_network_sorts(E, ties):
    rng = random.Random(E * 10 + ties)
    threads = 128  # four warps: strides of 32E and more still go through shared memory
    n = threads * E
    keys = [rng.choice((3, 5, 7)) if ties else rng.getrandbits(64) for _ in range(n)]
    assert _sort(keys, threads, E) == sorted(keys)


def test_swizzle_is_a_permutation_within_16_word_blocks():
    for w in range(1 << 14):
        assert _swz(w) >> 4 == w >> 4
    assert sorted(_swz(w) for w in range(8192)) == list(range(8192))


def test_swizzle_spreads_both_access_patterns():
    # 16 lanes of a 64-bit access (one phase) hit 16 distinct bank pairs, for
    # the blocked layout (lane l reads word l*E + j) and for contiguous words.
    for E in (2, 4, 8):
        for j in range(E):
            assert len({_swz(l * E + j) % 16 for l in range(16)}) == 16
    for base in range(0, 4096, 16):
        assert len({_swz(base + l) % 16 for l in range(16)}) == 16


def _sort_one(keys, P):
    """bitonic_one: the first P keys, one per thread; strides below 32 between
    lanes of a warp, 32 and more through shared memory."""
    mem = [0] * max(P, 1)
    v = list(keys[:P])
    size = 2
    while size <= P:
        stride = size >> 1
        if stride >= 32:
            for t in range(P):
                mem[_swz(t)] = v[t]
            while stride >= 32:
                for i in range(P // 2):
                    _cx_shared(mem, i, stride, size)
                stride >>= 1
            v = [mem[_swz(t)] for t in range(P)]
        while stride > 0:
            nv = list(v)
            for t in range(P):
                assert (t ^ stride) // 32 == t // 32 and (t ^ stride) < P
                o = v[t ^ stride]
                keep_min = ((t & stride) == 0) == ((t & size) == 0)
                nv[t] = min(o, v[t]) if keep_min else max(o, v[t])
            v = nv
            stride >>= 1
        size <<= 1
    return v


@pytest.mark.parametrize("P", [1, 2, 16, 32, 64, 256, 1024])
def test_one_key_per_thread_network_sorts(P):
    rng = random.Random(P)
    m = max(1, P - P // 3)  # padded like the kernel: keys past m are all ones
    keys = [rng.choice((3, 5, 7, 1 << 40)) for _ in range(m)] + [(1 << 64) - 1] * (P - m)
    assert _sort_one(keys, P) == sorted(keys)


def _f32_bits(x):
    import struct
    return struct.unpack("<I", struct.pack("<f", x))[0]


def _key(s, k, b):
    return ((0xFFFFFFFF - _f32_bits(max(s, 0.0))) << 32) | (k << 16) | b


def _select(surv, cap=1024, bins=1024):
    """The kernel's selection: histogram of float bits >> 20, thread t holds the
    count of bins >= bins - 1 - t, nfit = how many of those counts fit cap."""
    hist = [0] * bins
    for s in surv:
        hist[_f32_bits(min(max(s, 0.0), 1.0)) >> 20] += 1
    counts, acc = [], 0
    for t in range(bins):
        acc += hist[bins - 1 - t]
        counts.append(acc)
    nfit = sum(1 for c in counts if c <= cap)
    m_sel = counts[nfit - 1] if nfit else 0
    bin_lo = bins - nfit
    chosen = [i for i, s in enumerate(surv) if (_f32_bits(min(max(s, 0.0), 1.0)) >> 20) >= bin_lo]
    return m_sel, chosen


@pytest.mark.parametrize("B,K", [(128, 16), (512, 16), (256, 32), (4, 4), (1, 1)])
def test_selection_is_a_prefix_of_the_sorted_order(B, K):
    import numpy as np
    rng = np.random.default_rng(B * 100 + K)
    c = 1.0 / (1.0 + np.exp(-(3.0 + rng.normal(0, 2.0, size=(B, K))))).astype(np.float32)
    c[rng.random((B, K)) < 0.05] = 1.0  # exact ones make ties
    s = np.cumprod(c, axis=1, dtype=np.float32)
    surv = [float(x) for x in s.reshape(-1)]
    keys = [_key(surv[b * K + k], k, b) for b in range(B) for k in range(K)]
    m_sel, chosen = _select(surv)
    assert m_sel == len(chosen) <= 1024
    full = sorted(keys)
    assert sorted(keys[i] for i in chosen) == full[:m_sel]
    if B * K <= 1024:
        assert m_sel == B * K


def _merge_tree(a, off, Bp):
    """merge_tree: request b's run at off[b] .. off[b+1]; level l merges the runs
    of request groups 2j and 2j+1 of size 2^l by (own index) + (partner keys
    below), as the kernel does for every key at once."""
    m = off[Bp]
    l = 0
    while (1 << l) < Bp:
        t = [None] * m
        for i in range(m):
            x = a[i]
            g = (x & 0xFFFF) >> l
            own_lo = off[g << l]
            pg = g ^ 1
            lo, hi = off[pg << l], off[(pg + 1) << l]
            p_lo = lo
            while lo < hi:
                mid = (lo + hi) >> 1
                if a[mid] < x:
                    lo = mid + 1
                else:
                    hi = mid
            m_lo = off[(g >> 1) << (l + 1)]
            j = m_lo + (i - own_lo) + (lo - p_lo)
            assert t[j] is None
            t[j] = x
        a = t
        l += 1
    return a


@pytest.mark.parametrize("B,K", [(128, 16), (100, 8), (1, 4), (3, 2), (512, 16)])
def test_merge_tree_sorts_the_selected_runs(B, K):
    import numpy as np
    rng = np.random.default_rng(B + K)
    c = 1.0 / (1.0 + np.exp(-(2.0 + rng.normal(0, 2.0, size=(B, K))))).astype(np.float32)
    c[rng.random((B, K)) < 0.05] = 1.0
    s = np.cumprod(c, axis=1, dtype=np.float32)
    m_sel, chosen = _select([float(x) for x in s.reshape(-1)])
    # each request's selected positions form a prefix, laid out in request order
    Bp = 1
    while Bp < B:
        Bp <<= 1
    L = [0] * Bp
    for i in chosen:
        L[i // K] += 1
    for b in range(B):
        assert sorted(i % K for i in chosen if i // K == b) == list(range(L[b]))
    off = [0]
    for b in range(Bp):
        off.append(off[-1] + L[b])
    a = [_key(float(s[b, k]), k, b) for b in range(B) for k in range(L[b])]
    assert off[Bp] == m_sel == len(a)
    assert _merge_tree(a, off, Bp) == sorted(a)
