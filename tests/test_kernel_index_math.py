"""Model checks of kernels' index arithmetic, on the CPU.

compute-sanitizer is not available to this build, so the bounds and
coverage arguments the kernels rely on are checked here by enumerating
their index formulas over the shapes they run at: every element is touched
exactly once where a kernel partitions work, and every address stays inside
its buffer.  The formulas restate the kernels' own (decode.cu, backward.cu,
gdn_bwd_chunk.cu); a change there has to be mirrored here.
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


# ------------------------------- backward, chunkwise Gated DeltaNet adjoint
def _ldsm_rows_cols(kind, lane, m0, n0, j, k0):
    # the (row, column) of the fp16 tile a lane's ldmatrix address points to,
    # as in gdn_bwd_chunk.cu's hmm(): A stored [m][k] ("a") or [k][m] ("at"),
    # B stored [n][k] ("b") or [k][n] ("bt"); j = the first of two n8 tiles
    mi, r8 = lane >> 3, lane & 7
    if kind == "a":
        return m0 + (lane & 15), k0 + 8 * (lane >> 4)
    if kind == "at":
        return k0 + (mi >> 1) * 8 + r8, m0 + (mi & 1) * 8
    if kind == "b":
        return n0 + 8 * j + (mi >> 1) * 8 + r8, k0 + (mi & 1) * 8
    return k0 + (mi & 1) * 8 + r8, n0 + 8 * j + (mi >> 1) * 8


@pytest.mark.parametrize("D", [64, 128])
def test_chunk_adjoint_fragments_stay_in_their_tiles(D):
    # every product of the per-chunk kernels: output C x D (NT = D / 16, n0 =
    # (w >> 2) D / 2) or C x C (NT = 4, n0 = 32 (w >> 2)), m0 = 16 (w & 3),
    # over tiles of C x D, D x D or C x C fp16 entries, row stride cols + 8
    C = 64
    shapes = {"CD": (C, D), "DD": (D, D), "CC": (C, C)}
    products = [  # (output columns, K, A tile, A kind, B tile, B kind)
        (C, D, "CD", "a", "CD", "b"),    # K K^T, Q K^T, Y U^T, dO U^T
        (D, D, "CD", "a", "DD", "b"),    # dO S0, U dS_C, dVh S0 (S0, dS_C stored [dk][dv])
        (D, D, "CD", "a", "DD", "bt"),   # K S0^T, K~ dS_C^T
        (D, C, "CC", "a", "CD", "bt"),   # Linv diag(.) K, P W, Linv diag(beta) Vh, dPm K, A~ K
        (D, C, "CC", "at", "CD", "bt"),  # P^T dO, Linv^T dU, dPm^T Q, A~^T K
    ]
    for ncols, K, ta, ka, tb, kb in products:
        NT = ncols // 16 if ncols == D else 4
        seen_a, seen_b = set(), set()
        for w in range(8):
            m0, n0 = 16 * (w & 3), (w >> 2) * (ncols // 2)
            for k0 in range(0, K, 16):
                for lane in range(32):
                    r, c = _ldsm_rows_cols(ka, lane, m0, n0, 0, k0)
                    rows, cols = shapes[ta]
                    assert r < rows and c + 8 <= cols and (r * (cols + 8) + c) * 2 % 16 == 0
                    seen_a.add((r, c))
                    for j in range(0, NT, 2):
                        r, c = _ldsm_rows_cols(kb, lane, m0, n0, j, k0)
                        rows, cols = shapes[tb]
                        assert r < rows and c + 8 <= cols and (r * (cols + 8) + c) * 2 % 16 == 0
                        seen_b.add((r, c))
        # the product reads exactly its operands' 8-element row segments:
        # A over (C output rows) x K, B over K x (output columns)
        def segs(kind, nrows, ncols_):
            return {(r, c) for r in range(nrows) for c in range(0, ncols_, 8)}
        assert seen_a == (segs(0, C, K) if ka == "a" else segs(0, K, C)), (ncols, K, ka)
        assert seen_b == (segs(0, ncols, K) if kb == "b" else segs(0, K, ncols)), (ncols, K, kb)


def test_reverse_scan_transposed_store():
    """gdn_bwd_scan_kernel stores each committed chunk's dS_C rows (RB = 64 of
    them per CTA, fp32 shared rows of stride D + 4) transposed, four rows of
    one column per 16-byte store: every (row, column) exactly once, inside
    both buffers, 16-byte aligned, and each warp's stores four whole
    128-byte lines."""
    RB = 64
    for D in (64, 128):
        FS = D + 4
        seen = set()
        for w0 in range(0, RB * D // 4, 32):
            lines = set()
            for lane in range(32):
                x = w0 + lane
                b, l = x >> 5, x & 31
                i = 32 * (b % (RB // 32)) + 4 * (l & 7)
                kc = 4 * (b // (RB // 32)) + (l >> 3)
                assert 0 <= i <= RB - 4 and 0 <= kc < D
                assert ((i + 3) * FS + kc) < RB * FS
                off = kc * D + i  # floats from a 64-row-aligned base
                assert off % 4 == 0
                for j in range(4):
                    seen.add((i + j, kc))
                lines.add(off * 4 // 128)
            assert len(lines) == 4
        assert len(seen) == RB * D
