"""Address table of the attention kernel's cluster split, checked on the CPU.

The attention kernel runs one thread-block cluster per (unit, query row) with
ceil(K / 128) CTAs rounded up to a power of two; the merge gives each CTA
W = 512 / C output columns. This restates the kernel's index arithmetic for the
partial-output stores, the merge's bulk copies and the output stores, and
checks for every accepted K that each access is 16-byte aligned, stays inside
its buffer, and that every output element is produced exactly once. (A cluster
size that does not divide 512 would misalign the stores; the power-of-two
rounding is what rules that out.)
"""
import numpy as np

NC, MAX_CLUSTER, MAX_K = 128, 16, 2048
Y_BYTES = 9 * NC * 128          # the kernel's shared region that receives the merge copies


def cluster_ctas(K):
    need = (K + NC - 1) // NC
    C = 1
    while C < need:
        C *= 2
    return C


def test_cluster_size_for_every_accepted_k():
    for K in range(1, MAX_K + 1):
        C = cluster_ctas(K)
        assert C <= MAX_CLUSTER and C * NC >= K and (C == 1 or (C // 2) * NC < K)
        assert 512 % C == 0 and (512 // C) % 32 == 0
        rows = [max(0, min(NC, K - NC * c)) for c in range(C)]
        assert sum(rows) == K and all(r == NC for r in rows[:K // NC])


def partial_store_offsets(C):
    """Float offsets (within one CTA's 64 x 512 slot) written by the partial-O
    stores: warps 0, 1, 4, 5; 8 column blocks of 32; lanes store float4s."""
    W = 512 // C
    out = []
    for warp in (0, 1, 4, 5):
        q, c0 = warp & 3, 256 * (warp >> 2)
        for c in range(8):
            col = c0 + 32 * c
            blk = (col // W) * 64 * W + (col % W)
            for r4 in range(8):
                for lane in range(32):
                    r = 4 * r4 + (lane >> 3)
                    off = blk + (32 * q + r) * W + 4 * (lane & 7)
                    head, first_col = 32 * q + r, col + 4 * (lane & 7)
                    out.append((off, head, first_col))
    return out


def test_partial_output_stores_are_aligned_slice_major_and_complete():
    for C in (1, 2, 4, 8, 16):
        W = 512 // C
        seen = np.zeros(64 * 512, np.int32)
        for off, head, col in partial_store_offsets(C):
            assert off % 4 == 0 and 0 <= off and off + 4 <= 64 * 512
            # slice-major: column col of head h sits in slice col // W at [h][col % W]
            assert off == (col // W) * 64 * W + head * W + col % W
            seen[off:off + 4] += 1
        assert (seen == 1).all()


def test_merge_copies_and_output_stores():
    for C in (1, 2, 4, 8, 16):
        W = 512 // C
        blk_bytes = 64 * W * 4
        assert blk_bytes % 16 == 0 and C * blk_bytes <= Y_BYTES
        out = np.zeros((64, 512), np.int32)
        for crank in range(C):
            src = crank * 64 * W * 4                 # byte offset inside each source slot
            assert src % 16 == 0 and src + blk_bytes <= 64 * 512 * 4
            for c in range(C):
                assert (c * 64 * W * 4) % 16 == 0    # destination inside the shared buffer
            nq = W // 4
            for t in range(64 * nq):
                h, q4 = divmod(t, nq)
                col = crank * W + 4 * q4
                assert (h * 512 + col) % 4 == 0
                out[h, col:col + 4] += 1
        assert (out == 1).all()
