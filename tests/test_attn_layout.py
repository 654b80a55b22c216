"""Address table of the attention kernels' split, checked on the CPU.

The attention runs as two kernels. The first has ceil(K / 128) CTAs per
(unit, query row); CTA c computes the split-softmax part of selected rows
[128c, 128c + 128) and stores its 64 x 512 fp32 partial output slice-major
(16 slices of 32 columns, each a contiguous [64 heads][32] block) plus its 64
row maxima and sums. The second has one block per (unit, query row) and slice
and writes the final output. This restates both kernels' index arithmetic and
checks, for every accepted K, that each access is 16-byte aligned, stays
inside the workspace, that every partial element is stored exactly once, and
that every output element is produced exactly once from every part.
"""
import numpy as np

NC, MAX_CTAS, MAX_K = 128, 16, 2048
SLICE, NSLICE = 32, 16
PART_O, PART_ML = 64 * 512, 128


def attn_ctas(K):
    return (K + NC - 1) // NC


def workspace_floats(U, R):
    return U * R * MAX_CTAS * (PART_O + PART_ML)


def test_cta_count_and_row_ranges_for_every_accepted_k():
    for K in range(1, MAX_K + 1):
        C = attn_ctas(K)
        assert 1 <= C <= MAX_CTAS
        rows = [max(0, min(NC, K - NC * c)) for c in range(C)]
        assert sum(rows) == K and all(r > 0 for r in rows)
        assert all(r == NC for r in rows[:-1])


def partial_store_offsets():
    """Float offsets within one CTA's 64 x 512 slot written by the partial-O
    stores: all 8 warps; warp w reads tensor-memory lane quarter w & 3 (heads
    32 * (w & 1) + lane, lanes 64..127 repeating 0..63) and 128 columns from
    128 * (2 * (w >> 2) + ((w & 3) >> 1)); each 32 x 32 block is written as
    float4 runs of its slice."""
    out = []
    for warp in range(8):
        q = warp & 3
        hb = 32 * (q & 1)
        c0 = 128 * (2 * (warp >> 2) + (q >> 1))
        for c in range(4):
            col = c0 + 32 * c
            blk = (col // SLICE) * 64 * SLICE
            for r4 in range(8):
                for lane in range(32):
                    r = 4 * r4 + (lane >> 3)
                    off = blk + (hb + r) * SLICE + 4 * (lane & 7)
                    out.append((off, hb + r, col + 4 * (lane & 7)))
    return out


def test_partial_output_stores_are_aligned_slice_major_and_complete():
    seen = np.zeros(PART_O, np.int32)
    for off, head, col in partial_store_offsets():
        assert off % 4 == 0 and 0 <= off and off + 4 <= PART_O
        # slice-major: column col of head h sits in slice col // 32 at [h][col % 32]
        assert off == (col // SLICE) * 64 * SLICE + head * SLICE + col % SLICE
        seen[off:off + 4] += 1
    assert (seen == 1).all()


def test_part_slots_inside_the_workspace():
    for U, R in ((1, 1), (4, 1), (32, 1), (3, 4)):
        total = workspace_floats(U, R)
        o_end = U * R * MAX_CTAS * PART_O
        for ur in range(U * R):
            for c in range(MAX_CTAS):
                o = (ur * MAX_CTAS + c) * PART_O
                ml = o_end + (ur * MAX_CTAS + c) * PART_ML
                assert o % 4 == 0 and o + PART_O <= o_end
                assert ml % 4 == 0 and ml + PART_ML <= total


def test_merge_reads_every_part_and_writes_every_output_once():
    for K in (1, 128, 129, 300, 640, 1500, 2048):
        C = attn_ctas(K)
        out = np.zeros((64, 512), np.int32)
        for s in range(NSLICE):
            for t in range(64 * (SLICE // 4)):
                h, q4 = divmod(t, SLICE // 4)
                for c in range(C):
                    src = c * PART_O + s * 64 * SLICE + h * SLICE + 4 * q4
                    assert src % 4 == 0 and src + 4 <= MAX_CTAS * PART_O
                dst = h * 512 + s * SLICE + 4 * q4
                assert dst % 4 == 0
                out[h, s * SLICE + 4 * q4:s * SLICE + 4 * q4 + 4] += 1
        assert (out == 1).all()
