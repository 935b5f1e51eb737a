"""Model checks of kernels' index arithmetic, on the CPU.

compute-sanitizer is not available to this build, so the bounds and
coverage arguments the kernels rely on are checked here by enumerating
their index formulas over the shapes they run at: every element is touched
exactly once where a kernel partitions work, and every address stays inside
its buffer.  The formulas restate the kernels' own (decode.cu, backward.cu,
backward_mma.cu); a change there has to be mirrored here.
"""

import itertools

import pytest

C = 64  # chunk


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("D,elem", [(128, 2), (128, 4), (64, 2), (64, 4)])
def test_decode_key_blocks_cover_each_key_once(D, elem):
    # decode_step_kernel: the hi = nr + p keys held in memory (nr retained,
    # p of the current chunk) in blocks of 32 claimed by the cluster's CTAs;
    # block b copies rows [32 b, min(32 b + 32, hi)) as a retained run and a
    # chunk run; warp w of the CTA scores stage rows 8 w .. 8 w + 7
    kps, row = 32, D * elem
    for nr in range(0, 64 * 33, 64):
        for p in (0, 1, 31, 32, 33, 63):
            hi, cap = nr + p, nr + 64
            seen = [0] * hi
            for b in range((hi + kps - 1) // kps):
                a0, a1 = b * kps, min(b * kps + kps, hi)
                m = min(max(nr, a0), a1)
                assert 0 < a1 - a0 <= kps
                if m > a0:
                    assert m <= nr <= cap  # retained rows exist
                if a1 > m:
                    assert 0 <= m - nr and a1 - nr <= p < C  # chunk rows before the token
                for run in (m - a0, a1 - m):
                    assert run * row % 16 == 0  # bulk-copy size
                assert (a1 - a0) * row <= kps * row  # fits the stage
                for w in range(4):
                    for u in range(8):
                        j = b * kps + 8 * w + u
                        if j < hi:
                            assert 8 * w + u < a1 - a0  # a landed row
                            seen[j] += 1
            assert all(c == 1 for c in seen), (nr, p)


def test_decode_state_rows_and_chunk_append_split():
    # every CTA of the cluster of 8 owns d / 8 state rows (TPR threads per
    # row, CPT columns each) and 8 of the chunk's 64 rows to append
    for D in (64, 128):
        rpc, threads, k_split = D // 8, 128, 8
        tpr = threads // rpc
        cpt = D // tpr
        seen = set()
        for rank in range(k_split):
            for tid in range(threads):
                row, part = rank * rpc + tid // tpr, tid % tpr
                for j in range(cpt):
                    key = (row, part * cpt + j)
                    assert key not in seen and row < D and part * cpt + j < D
                    seen.add(key)
        assert len(seen) == D * D
        rows = sorted(rank * 8 + e // D for rank in range(k_split) for e in range(8 * D) if e % D == 0)
        assert rows == list(range(C))


# --------------------------------------------------- backward, Gated DeltaNet
@pytest.mark.parametrize("D", [64, 128])
def test_backward_adjoint_covers_the_state_once(D):
    # gdn_bwd_kernel: two CTAs per head own rows [part RH, part RH + RH);
    # thread (warp, lane) holds rows warp RW + i and columns lane CW + j
    split, warps = 2, 16
    rh, cw = D // split, D // 32
    rw = rh // warps
    seen = set()
    for part, warp, lane in itertools.product(range(split), range(warps), range(32)):
        for i, j in itertools.product(range(rw), range(cw)):
            r, c = part * rh + warp * rw + i, lane * cw + j
            assert 0 <= r < D and 0 <= c < D and (r, c) not in seen
            seen.add((r, c))
    assert len(seen) == D * D
    # the token-vector slots: k, scale q (D each), v and do of the CTA's rows, a, beta
    tok = 2 * D + 2 * rh + 2
    assert tok <= 512


def test_backward_partials_match_between_writer_and_combine():
    # writer: pcol + ((part * BH + bh) * L + t) * 2 D; combine: pcol + ((h * rows
    # + r) * 2 D) with rows = BH L and r = bh L + t: the same element
    for BH, L, D in ((3, 128, 64), (4, 256, 128)):
        rows = BH * L
        for part, bh, t in itertools.product(range(2), range(BH), (0, 1, L - 1)):
            writer = ((part * BH + bh) * L + t) * 2 * D
            combine = (part * rows + (bh * L + t)) * 2 * D
            assert writer == combine
            assert writer + 2 * D <= 2 * rows * 2 * D  # inside the buffer of both shares


# ------------------------------------------- backward, tensor-core softmax
def _frag_rows_cols(kind, lane, a, b):
    # the (row, column) a lane's ldmatrix address points to, as in
    # backward_mma.cu: frag_a (m0 = a, ks = b), frag_bt (jp = a, ks = b),
    # frag_b (ks = a, np = b)
    if kind == "a":
        return a + (lane & 7) + 8 * ((lane >> 3) & 1), 16 * b + 8 * (lane >> 4)
    if kind == "bt":
        return 16 * a + (lane & 7) + 8 * (lane >> 4), 16 * b + 8 * ((lane >> 3) & 1)
    return 16 * a + (lane & 7) + 8 * ((lane >> 3) & 1), 16 * b + 8 * (lane >> 4)


@pytest.mark.parametrize("D", [64, 128])
def test_backward_mma_fragments_stay_in_their_tiles(D):
    rs = D + 8  # skewed row stride; a lane reads 8 bf16 (16 bytes) from its address
    for lane in range(32):
        for m0 in range(0, 64, 16):
            for ks in range(D // 16):  # A over the feature dimension (Q, dO, K, V rows)
                r, c = _frag_rows_cols("a", lane, m0, ks)
                assert r < 64 and c + 8 <= D and (r * rs + c) * 2 % 16 == 0
        for jp in range(4):
            for ks in range(D // 16):  # K^T / V^T / Q^T / dO^T operands
                r, c = _frag_rows_cols("bt", lane, jp, ks)
                assert r < 64 and c + 8 <= D and (r * rs + c) * 2 % 16 == 0
        for ks in range(4):
            for np_ in range(D // 16):  # K / dO / Q as [k][n] operands
                r, c = _frag_rows_cols("b", lane, ks, np_)
                assert r < 64 and c + 8 <= D and (r * rs + c) * 2 % 16 == 0
