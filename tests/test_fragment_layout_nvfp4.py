"""The operand layout of the NVFP4-cache decode's warp-level products, checked
on the CPU (the arithmetic of the layout, not of the kernel).

An m16n8k16 product with fp16 operands takes, in lane (g, q) = (lane / 4,
lane % 4): A registers R0 = (row g, columns 2q, 2q + 1), R1 = (row g + 8, the
same columns), R2 = (row g, columns 2q + 8, 2q + 9), R3 = (row g + 8, those
columns); B registers b0 = (rows 2q, 2q + 1, column g), b1 = (rows 2q + 8,
2q + 9, column g); and returns C registers c0, c1 = (row g, columns 2q,
2q + 1), c2, c3 = (row g + 8, the same columns).

The score warps give lane (g, q), in k-step kk, the key elements
32q + 4kk + {0, 1} as columns 2q, 2q + 1 and 32q + 4kk + {2, 3} as columns
2q + 8, 2q + 9, and the query head g's same elements as B.  Summed over the
eight k-steps this must be the plain S = K Q^T of the 16 keys: a permutation
of the contracted dimension that A and B share.  The code bytes a lane reads
(16q .. 16q + 15 of each row) and the block scales it applies (2q for
k-steps 0-3, 2q + 1 for 4-7) are checked to be the ones its elements need.
"""
import numpy as np


def mma16816(A_regs, B_regs):
    """Emulate one warp's m16n8k16 product from per-lane fragments:
    A_regs[lane] = 4 pairs, B_regs[lane] = 2 pairs -> C_regs[lane] = 4."""
    A = np.zeros((16, 16))
    B = np.zeros((16, 8))
    for lane in range(32):
        g, q = lane // 4, lane % 4
        r0, r1, r2, r3 = A_regs[lane]
        A[g, 2 * q:2 * q + 2] = r0
        A[g + 8, 2 * q:2 * q + 2] = r1
        A[g, 2 * q + 8:2 * q + 10] = r2
        A[g + 8, 2 * q + 8:2 * q + 10] = r3
        b0, b1 = B_regs[lane]
        B[2 * q:2 * q + 2, g] = b0
        B[2 * q + 8:2 * q + 10, g] = b1
    C = A @ B
    out = []
    for lane in range(32):
        g, q = lane // 4, lane % 4
        out.append((C[g, 2 * q], C[g, 2 * q + 1], C[g + 8, 2 * q], C[g + 8, 2 * q + 1]))
    return out


def test_permuted_k_steps_give_the_plain_product():
    rng = np.random.default_rng(7)
    K = rng.standard_normal((16, 128))  # 16 keys (one product's rows) x d
    Q = rng.standard_normal((8, 128))   # 8 head columns (heads past G are zero rows)
    S = np.zeros((16, 8))
    for kk in range(8):
        A_regs, B_regs = [], []
        for lane in range(32):
            g, q = lane // 4, lane % 4
            e = 32 * q + 4 * kk
            A_regs.append((K[g, e:e + 2], K[g + 8, e:e + 2], K[g, e + 2:e + 4],
                           K[g + 8, e + 2:e + 4]))
            B_regs.append((Q[g, e:e + 2], Q[g, e + 2:e + 4]))
        C = mma16816(A_regs, B_regs)
        for lane in range(32):
            g, q = lane // 4, lane % 4
            S[g, 2 * q:2 * q + 2] += C[lane][0:2]
            S[g + 8, 2 * q:2 * q + 2] += C[lane][2:4]
    np.testing.assert_allclose(S, K @ Q.T, rtol=1e-12, atol=1e-12)


def test_a_lane_reads_its_own_bytes_and_scales():
    """Every element a lane feeds lies in code bytes 16q .. 16q + 15 of its
    rows (two per byte, element 2i in the low nibble), in word kk / 2 of
    those 16 bytes, and its block scale is 2q for k-steps 0-3, 2q + 1 after;
    over the four lanes of a row group the 128 elements are fed once each."""
    for g in range(8):
        seen = []
        for q in range(4):
            for kk in range(8):
                for off in range(4):
                    e = 32 * q + 4 * kk + off
                    byte = e // 2
                    assert 16 * q <= byte < 16 * q + 16
                    assert (byte - 16 * q) // 4 == kk // 2          # word of the 16-byte load
                    assert (byte - 16 * q) % 4 == 2 * (kk % 2) + off // 2  # byte in the word
                    assert e // 16 == 2 * q + (kk >= 4)             # block scale index
                    seen.append(e)
        assert sorted(seen) == list(range(128))


def test_value_fragments_from_the_transposed_loads():
    """O^T += V^T P^T: lane l of an x4 transposed load gives row l % 8 of
    matrix l / 8 (keys + 8 for matrices 2, 3; value dimensions + 8 for
    matrices 1, 3); a transposed 8 x 8 load hands lane (g, q) the elements
    (rows 2q, 2q + 1, column g) of the stored matrix.  With the stored rows
    being keys and its columns value dimensions, the four registers must be
    the A fragment of V^T (rows = dimensions, columns = keys), and the P^T
    rows loaded untransposed (rows = heads, 8 keys each) the B fragment."""
    rng = np.random.default_rng(11)
    V = rng.standard_normal((16, 16))   # 16 keys x 16 value dimensions of one product
    P = rng.standard_normal((8, 16))    # 8 heads x 16 keys
    A_regs, B_regs = [], []
    for lane in range(32):
        g, q = lane // 4, lane % 4
        regs = []
        for m in range(4):  # matrix m: keys 8 (m >> 1) .., dimensions 8 (m & 1) ..
            k0, d0 = 8 * (m >> 1), 8 * (m & 1)
            tile = V[k0:k0 + 8, d0:d0 + 8]        # stored rows = keys
            regs.append(tile[2 * q:2 * q + 2, g])  # the transposed load's pair
        A_regs.append(tuple(regs))
        b = []
        for m in range(2):  # untransposed: rows = heads, keys 8m ..
            tile = P[:, 8 * m:8 * m + 8]
            b.append(tile[g, 2 * q:2 * q + 2])
        B_regs.append(tuple(b))
    C = mma16816(A_regs, B_regs)
    OT = V.T @ P.T  # [dimensions, heads]
    for lane in range(32):
        g, q = lane // 4, lane % 4
        np.testing.assert_allclose(C[lane], (OT[g, 2 * q], OT[g, 2 * q + 1],
                                             OT[g + 8, 2 * q], OT[g + 8, 2 * q + 1]),
                                   rtol=1e-12, atol=1e-12)


def test_a_swapped_register_pair_is_caught():
    """Self-check: R1 and R2 swapped (row g + 8 and the upper columns
    confused) must not reproduce the product."""
    rng = np.random.default_rng(5)
    K = rng.standard_normal((16, 16))
    Q = rng.standard_normal((8, 16))
    A_regs, B_regs = [], []
    for lane in range(32):
        g, q = lane // 4, lane % 4
        A_regs.append((K[g, 2 * q:2 * q + 2], K[g, 2 * q + 8:2 * q + 10],
                       K[g + 8, 2 * q:2 * q + 2], K[g + 8, 2 * q + 8:2 * q + 10]))
        B_regs.append((Q[g, 2 * q:2 * q + 2], Q[g, 2 * q + 8:2 * q + 10]))
    C = mma16816(A_regs, B_regs)
    S = K @ Q.T
    got = np.array([[C[4 * g + q][0], C[4 * g + q][1]] for g in range(8) for q in range(4)])
    want = np.array([[S[g, 2 * q], S[g, 2 * q + 1]] for g in range(8) for q in range(4)])
    assert not np.allclose(got, want)
