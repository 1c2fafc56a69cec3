"""The fragment layouts of the decode's tensor-core slices, emulated lane by lane on
the CPU (no GPU, no library code). The kernel builds its m16n8k16 operands so that
every lane reads whole pieces of shared memory with no shuffles, which requires
permuting the head dims inside a k-step and the rows of O^T; these tests rebuild the
A / B / C matrices from the per-lane fragment contents exactly as the PTX ISA defines
the m16n8k16 .row.col layout, and check that the products equal q . k and p . v for
both cache formats (bf16 rows; 4-bit codes, K placed under fp16 magic exponents as the
rows of S^T = K Q^T, V as fp16 subnormals), and that the 8 x 8 transposes turn the
4-bit path's scores into its P^T fragments."""

import numpy as np
import pytest

LANES = [(l >> 2, l & 3) for l in range(32)]  # (gid, tig)


def mma(afr, bfr):
    """C (16 x 8) = A (16 x 16) B (16 x 8) from per-lane fragments: afr[lane] =
    (a0, a1, a2, a3), each a pair (low, high) of values; bfr[lane] = (b0, b1)."""
    A = np.full((16, 16), np.nan)
    B = np.full((16, 8), np.nan)
    for lane, (g, t) in enumerate(LANES):
        a0, a1, a2, a3 = afr[lane]
        for e in range(2):
            A[g, 2 * t + e], A[g + 8, 2 * t + e] = a0[e], a1[e]
            A[g, 2 * t + 8 + e], A[g + 8, 2 * t + 8 + e] = a2[e], a3[e]
        b0, b1 = bfr[lane]
        for e in range(2):
            B[2 * t + e, g], B[2 * t + 8 + e, g] = b0[e], b1[e]
    assert not np.isnan(A).any() and not np.isnan(B).any()
    C = A @ B
    return [((C[g, 2 * t], C[g, 2 * t + 1]), (C[g + 8, 2 * t], C[g + 8, 2 * t + 1])) for g, t in LANES]


def half_bits_value(bits):
    return float(np.array([bits], np.uint16).view(np.float16)[0])


def fp16_pair(word):
    return half_bits_value(word & 0xFFFF), half_bits_value(word >> 16)


def v_group_bytes(codes, D):
    """The 4-bit V layout of one 16-row group as include/duo_attn.h states it: the byte of
    row k and dims (2 dp, 2 dp + 1) (low, high nibble) at 4 ((4 (dp / MT) + (k % 8) / 2)
    MT + dp % MT) + 2 (k % 2) + k / 8, MT = D / 16."""
    MT = D // 16
    out = np.full(16 * D // 2, -1, np.int64)
    for k in range(16):
        for dp in range(D // 2):
            a = 4 * ((4 * (dp // MT) + (k % 8) // 2) * MT + dp % MT) + 2 * (k % 2) + k // 8
            assert out[a] < 0  # each byte holds one row's pair of codes
            out[a] = codes[k, 2 * dp] | (codes[k, 2 * dp + 1] << 4)
    assert (out >= 0).all()
    return out.astype(np.uint8)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_bf16_scores(D, G):
    """S = Q K^T: lane tig takes 16-byte chunk tig + 4u of a row, i.e. k-index 2 tig + i
    (+ 8) of k-step 2u + e is dim 8 (tig + 4u) + 4e + i (+ 2)."""
    rng = np.random.default_rng(D + G)
    q = rng.standard_normal((G, D))
    k = rng.standard_normal((16, D))
    S = np.zeros((G, 16))
    for j in range(2):  # n-tiles: keys gid, gid + 8
        acc = np.zeros((16, 8))
        for s in range(D // 16):
            u, e = divmod(s, 2)
            afr, bfr = [], []
            for g, t in LANES:
                c = t + 4 * u
                d = [8 * c + 4 * e + i for i in range(4)]  # the chunk's words 2e and 2e + 1
                qrow = q[g] if g < G else np.zeros(D)
                afr.append(((qrow[d[0]], qrow[d[1]]), (0, 0), (qrow[d[2]], qrow[d[3]]), (0, 0)))
                krow = k[g + 8 * j]
                bfr.append(((krow[d[0]], krow[d[1]]), (krow[d[2]], krow[d[3]])))
            out = mma(afr, bfr)
            for lane, (g, t) in enumerate(LANES):
                (c0, c1), _ = out[lane]
                acc[g, 2 * t] += c0
                acc[g, 2 * t + 1] += c1
        S[:, 8 * j:8 * j + 8] = acc[:G]
    assert np.allclose(S, q @ k.T)


def transpose8x8(frags):
    """movmatrix.m8n8.trans.b16 as the PTX ISA defines it: lane (gid, tig) holds row gid,
    cols 2 tig and 2 tig + 1 of an 8 x 8 matrix; afterwards the same of its transpose."""
    M = np.full((8, 8), np.nan)
    for lane, (g, t) in enumerate(LANES):
        M[g, 2 * t], M[g, 2 * t + 1] = frags[lane]
    assert not np.isnan(M).any()
    return [(M.T[g, 2 * t], M.T[g, 2 * t + 1]) for g, t in LANES]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_kv4_scores_keys_as_rows(D, G):
    """4-bit K, S^T = K Q^T: word w = (D/32) tig + u of a row holds dims 8w ... 8w+7
    (nibble n = dim 8w + n); k-index 2 tig + i (+ 8) of k-step 2u + e is dim 8w + 2e + 4i
    (+ 1); the A fragments are the words of keys gid and gid + 8 with the codes read as
    1024 + c (bits 0-3) or 64 + c (bits 4-7), the B fragment is head gid's q (zero for
    heads >= G); lane (gid, tig) gets keys gid, gid + 8 of heads 2 tig, 2 tig + 1, and
    S - sum_d q_d off_d = q . c."""
    rng = np.random.default_rng(D + G)
    q = np.zeros((8, D))
    q[:G] = np.round(rng.standard_normal((G, D)) * 64) / 64  # exact in fp16
    codes = rng.integers(0, 16, (16, D))
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)  # [16, D/2]
    words = np.ascontiguousarray(packed).view("<u4")  # [16, D/8]: word w = bytes 4w ... 4w+3
    WPT = D // 32
    lo, hi = 0x64006400, 0x54005400
    acc = np.zeros((16, 8))  # [key][head]
    for s in range(D // 16):
        u, e = divmod(s, 2)
        afr, bfr = [], []
        for g, t in LANES:
            w = WPT * t + u
            xa, xb = int(words[g, w]) >> (8 * e), int(words[g + 8, w]) >> (8 * e)
            afr.append((fp16_pair((xa & 0x000F000F) | lo), fp16_pair((xb & 0x000F000F) | lo),
                        fp16_pair((xa & 0x00F000F0) | hi), fp16_pair((xb & 0x00F000F0) | hi)))
            dims = [8 * w + 2 * e + 4 * i for i in range(2)]  # k = 2 tig + i
            dims8 = [d + 1 for d in dims]                       # k = 2 tig + 8 + i
            bfr.append(((q[g, dims[0]], q[g, dims[1]]), (q[g, dims8[0]], q[g, dims8[1]])))
        out = mma(afr, bfr)
        for lane, (g, t) in enumerate(LANES):
            (c0, c1), (c2, c3) = out[lane]
            acc[g, 2 * t] += c0
            acc[g, 2 * t + 1] += c1
            acc[g + 8, 2 * t] += c2
            acc[g + 8, 2 * t + 1] += c3
    off = (q[:, 0::2] * 1024).sum(1) + (q[:, 1::2] * 64).sum(1)
    assert np.allclose(acc - off[None, :], codes @ q.T)


def test_kv4_p_transpose_gives_the_pt_fragments():
    """The scores of a 16-key group sit in lanes as (key gid or gid + 8; heads 2 tig, 2 tig
    + 1); packing the pair of heads per key and transposing each 8 x 8 half gives the P^T
    fragment of O^T += V^T P^T: head gid's p of keys 2 tig, 2 tig + 1 (b0) and 2 tig + 8,
    2 tig + 9 (b1)."""
    p = np.random.default_rng(5).random((8, 16))  # [head][key]
    b0 = transpose8x8([(p[2 * t, g], p[2 * t + 1, g]) for g, t in LANES])
    b1 = transpose8x8([(p[2 * t, g + 8], p[2 * t + 1, g + 8]) for g, t in LANES])
    for lane, (g, t) in enumerate(LANES):
        assert b0[lane] == (p[g, 2 * t], p[g, 2 * t + 1])
        assert b1[lane] == (p[g, 2 * t + 8], p[g, 2 * t + 9])


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("kv4", [False, True])
def test_output_rows(D, G, kv4):
    """O^T += V^T P^T: m-tile i, row gid (gid + 8) is dim (D/8) gid + 2i (+ 1); the P^T
    fragment of lane (gid, tig) holds head gid's p of keys 2 tig, 2 tig + 1, 2 tig + 8,
    2 tig + 9; every (head < G, dim) comes out of exactly one lane and fragment slot."""
    rng = np.random.default_rng(D * G + kv4)
    DT = D // 8
    p = rng.random((8, 16))
    p[G:] = 0
    if kv4:
        codes = rng.integers(0, 16, (16, D))
        words = v_group_bytes(codes, D).view("<u4")  # the group's 32-bit words
        V = codes.astype(float)
    else:
        V = rng.standard_normal((16, D))
    O = np.full((G, D), np.nan)
    kr = lambda t: [2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9]
    for i in range(D // 16):
        afr, bfr = [], []
        for g, t in LANES:
            k0, k1, k2, k3 = kr(t)
            if kv4:
                # word i of lane (g, t): bytes = keys 2t, 2t + 8, 2t + 1, 2t + 9 (low nibble
                # dim d, high nibble dim d + 1); the shift by 8 brings keys 2t + 1, 2t + 9
                # down. The codes are fp16 subnormals: c 2^-24 (bits 0-3, even dims) and
                # c 2^-20 (bits 4-7, odd dims), scaled back per output dim below.
                w = int(words[(4 * g + t) * (D // 16) + i])
                x8 = w >> 8
                a0 = fp16_pair(w & 0x000F000F)
                a1 = fp16_pair(w & 0x00F000F0)
                a2 = fp16_pair(x8 & 0x000F000F)
                a3 = fp16_pair(x8 & 0x00F000F0)
            else:
                d0 = DT * g + 2 * i
                a0, a1 = (V[k0, d0], V[k1, d0]), (V[k0, d0 + 1], V[k1, d0 + 1])
                a2, a3 = (V[k2, d0], V[k3, d0]), (V[k2, d0 + 1], V[k3, d0 + 1])
            afr.append((a0, a1, a2, a3))
            bfr.append(((p[g, k0], p[g, k1]), (p[g, k2], p[g, k3])))
        out = mma(afr, bfr)
        for lane, (g, t) in enumerate(LANES):
            (c0, c1), (c2, c3) = out[lane]
            d = DT * g + 2 * i
            for h, (v_even, v_odd) in ((2 * t, (c0, c2)), (2 * t + 1, (c1, c3))):
                if kv4:
                    v_even, v_odd = v_even * 2.0 ** 24, v_odd * 2.0 ** 20
                if h < G:
                    assert np.isnan(O[h, d]) and np.isnan(O[h, d + 1])
                    O[h, d], O[h, d + 1] = v_even, v_odd
    assert not np.isnan(O).any()
    assert np.allclose(O, p[:G] @ V)
