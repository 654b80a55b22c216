"""Address table of the attention kernels, checked on the CPU.

The first kernel cuts the K selected rows of a (unit, query row) into chunks
of 64 and the chunks into at most 16 contiguous runs, one CTA per run; a CTA
keeps the query block and a 64-row fp16 tile in shared memory, stages the raw
rows of a chunk with one bulk copy (or, with the gather fused in, one bulk
copy per row from its source), and stores its unnormalised 64 x 512 fp32
output slice-major (16 slices of 32 columns, each a contiguous [64 heads][32]
block) plus its 64 row maxima and sums. The second kernel has one block per
(unit, query row) and slice. This restates the kernels' index arithmetic and
checks, for every accepted K and several batch sizes, that the runs cover the
chunks exactly once, that every shared-memory operand read of the tensor-core
products stays inside its region, that each store is 16-byte aligned and
inside the workspace, and that every output element is produced exactly once.
"""
import numpy as np

NC, MAX_CTAS, MAX_K = 64, 16, 2048
SLICE, NSLICE = 32, 16
PART_O, PART_ML = 64 * 512, 128
QATOM = 64 * 128
Q_OFF, T_OFF = 0, 9 * QATOM
P_OFF, R_OFF = T_OFF + 8 * QATOM, T_OFF + 9 * QATOM
MISC_OFF = R_OFF + NC * 656


def runs(K, UR, sms=152):
    """(chunks per run, runs) as the launch chooses them."""
    nchunks = (K + NC - 1) // NC
    want = min(max(1, sms // UR), nchunks, MAX_CTAS)
    cpp = (nchunks + want - 1) // want
    return cpp, (nchunks + cpp - 1) // cpp


def test_runs_cover_every_chunk_once():
    for UR in (1, 2, 4, 16, 32, 64, 200):
        for K in range(1, MAX_K + 1, 7):
            cpp, parts = runs(K, UR)
            nchunks = (K + NC - 1) // NC
            assert 1 <= parts <= MAX_CTAS
            seen = np.zeros(nchunks, int)
            for part in range(parts):
                c0, c1 = part * cpp, min(part * cpp + cpp, nchunks)
                assert c0 < c1
                seen[c0:c1] += 1
            assert (seen == 1).all()
            rows = [min(NC, K - NC * c) for c in range(nchunks)]
            assert sum(rows) == K and all(r > 0 for r in rows)


def sw128(row, k):
    return (row >> 3) * 1024 + (row & 7) * 128 + ((((k >> 3) ^ row) & 7) << 4) + (k & 7) * 2


def test_operand_spans_stay_inside_their_regions():
    # S = Q K^T: A = query atom kb read as M = 128 rows (16 groups of 1024 B;
    # the descriptor's 32-byte steps along K stay inside each 128-byte row);
    # B = tile atom kb, N = 64 rows (8 groups)
    for kb in range(9):
        a_atom = Q_OFF + kb * QATOM
        assert a_atom + 16 * 1024 <= MISC_OFF            # padded rows stay in shared memory
        b_atom = T_OFF + kb * QATOM
        assert b_atom + 8 * 1024 <= T_OFF + 9 * QATOM
        for kk in range(4):
            assert kk * 32 + 32 <= 128
    # O^T += V^T P^T: A = latent atoms 2mb, 2mb + 1 (MN-major, LBO = one atom),
    # 16 rows per product (2 groups); B = P, 64 heads (8 groups)
    for mb in range(4):
        for kk in range(NC // 16):
            a0 = T_OFF + 2 * mb * QATOM + kk * 2048
            assert a0 + QATOM + 2048 <= P_OFF              # never the RoPE / P atom
    assert P_OFF + 8 * 1024 <= R_OFF and (NC // 16 - 1) * 32 + 32 <= 128
    # the dequantised items and P rows
    for j in range(NC):
        for c in range(36):
            d0 = 16 * c
            for half in (0, 8):   # two 16-byte stores (the swizzle separates them)
                off = T_OFF + (d0 >> 6) * QATOM + sw128(j, (d0 & 63) + half)
                assert off % 16 == 0 and T_OFF <= off and off + 16 <= R_OFF
    for hd in range(64):
        for rh in range(2):
            for q4 in range(4):
                off = P_OFF + sw128(hd, 32 * rh + 8 * q4)
                assert off % 16 == 0 and P_OFF <= off < R_OFF


def partial_store_offsets():
    """Float offsets within one run's 64 x 512 slot written by the partial-O
    stores: warp w, lane l hold latent dim 128 mb + 32 (w & 3) + l of blocks
    mb = 2 (w >> 2) + b; per head the warp stores 32 consecutive floats."""
    out = []
    for warp in range(8):
        for b in range(2):
            mb = 2 * (warp >> 2) + b
            blk = (4 * mb + (warp & 3)) * 64 * SLICE
            for x2 in range(2):
                for k in range(32):
                    for lane in range(32):
                        d = 128 * mb + 32 * (warp & 3) + lane
                        out.append((blk + (32 * x2 + k) * SLICE + lane, 32 * x2 + k, d))
    return out


def test_partial_output_stores_are_slice_major_and_complete():
    seen = np.zeros(PART_O, np.int32)
    for off, head, d in partial_store_offsets():
        assert 0 <= off < PART_O
        assert off == (d // SLICE) * 64 * SLICE + head * SLICE + d % SLICE
        seen[off] += 1
    assert (seen == 1).all()


def test_merge_reads_every_run_and_writes_every_output_once():
    for K in (1, 64, 65, 300, 640, 1500, 2048):
        _, C = runs(K, 4)
        out = np.zeros((64, 512), np.int32)
        for s in range(NSLICE):
            for t in range(64 * (SLICE // 4)):
                h, q4 = divmod(t, SLICE // 4)
                for c in range(C):
                    src = c * PART_O + s * 64 * SLICE + h * SLICE + 4 * q4
                    assert src % 4 == 0 and src + 4 <= MAX_CTAS * PART_O
                out[h, s * SLICE + 4 * q4:s * SLICE + 4 * q4 + 4] += 1
        assert (out == 1).all()


def test_runs_follow_the_streams_sms():
    """On an SM partition the runs fill the partition's SMs (the launch
    passes the stream's SM count): fewer, longer runs, still every chunk once."""
    for sms in (32, 40, 48, 120, 152):
        for UR in (1, 16, 32):
            for K in (64, 2048, 1500, 300):
                cpp, parts = runs(K, UR, sms)
                nchunks = (K + NC - 1) // NC
                assert parts * UR <= max(UR, sms) or parts == 1
                assert (parts - 1) * cpp < nchunks <= parts * cpp


def test_gathered_row_copies_stay_in_the_staging_region():
    """The fused gather stages a chunk with one bulk copy per row: row j of
    the chunk lands at R_OFF + 656 j, 16-byte aligned, 656 bytes (a multiple
    of 16), and the 64 rows end where the next region begins."""
    assert 656 % 16 == 0 and R_OFF % 16 == 0
    for j in range(NC):
        dst = R_OFF + 656 * j
        assert dst % 16 == 0
        assert R_OFF <= dst and dst + 656 <= MISC_OFF
    # a source row p of a mirror, slot or ring array is 16-byte aligned when
    # the array is (the kernels skip units whose arrays are not)
    for p in (0, 1, 2, 3, 1048575):
        assert (656 * p) % 16 == 0
