"""The scheduler's sort network, restated on the host (no GPU).

schedule_kernel sorts n_pad = E * threads keys with each thread holding E
consecutive keys in registers: strides below E are exchanged in registers,
strides E .. 32E - 1 between the lanes of a warp, and strides of 32E and more
through shared memory, whose word w sits at w ^ ((w >> 4) & 15). This model
runs the same stages with the same index arithmetic (at fewer threads, which
keeps all three kinds of stage) and checks that the keys come out sorted and
that every lane partner lies in the same warp.
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
