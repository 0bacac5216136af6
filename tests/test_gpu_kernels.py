"""Each device kernel, through the C ABI, against the fp64 oracle (or exact bytes)."""
import numpy as np
import pytest
import torch

from host_offloaded_weight_gb300 import lstream as L
from oracle import forward as F

from gpu_util import rand_bf16, bf16_dev, to_f64, rel_err

pytestmark = pytest.mark.gpu


def _no_device_error():
    assert L.lsk_device_error() == 0


# ------------------------------------------------------------------ copy + hand-off
@pytest.mark.parametrize("nbytes", [1, 15, 16, 17, 4099, 65536 * 3 + 5, 10 * 2**20 + 7, 64 * 2**20])
@pytest.mark.parametrize("ctas", [1, 7, 0])
def test_copy_kernel_exact_bytes_and_publish(nbytes, ctas):
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8).pin_memory()
    dst = torch.zeros(nbytes + 64, dtype=torch.uint8, device="cuda")
    ready = torch.zeros(1, dtype=torch.int32, device="cuda")
    ticket = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.lsk_copy_h2slot(dst, src, nbytes, ctas, ready, ticket, 77)
    torch.cuda.synchronize()
    assert torch.equal(dst[:nbytes].cpu(), src)
    assert int(dst[nbytes:].abs().sum()) == 0, "wrote past the end"
    assert int(ready) == 77 and int(ticket) == 0


def test_copy_kernel_rejects_unpinned_and_unaligned():
    dst = torch.zeros(64, dtype=torch.uint8, device="cuda")
    w = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(L.LsError):
        L.lsk_copy_h2slot(dst, torch.zeros(64, dtype=torch.uint8), 64, 1, w, w[1:], 1)
    pinned = torch.zeros(80, dtype=torch.uint8).pin_memory()
    with pytest.raises(L.LsError):
        L.lsk_copy_h2slot(dst, pinned.data_ptr() + 4, 16, 1, w, w[1:], 1)


def test_wait_ready_passes_and_times_out():
    ready = torch.zeros(1, dtype=torch.int32, device="cuda")
    ticket = torch.zeros(1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32).pin_memory()
    src = torch.arange(4096, dtype=torch.uint8).pin_memory()
    dst = torch.empty(4096, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        L.lsk_copy_h2slot(dst, src, 4096, 4, ready, ticket, 5, stream=s)
        L.lsk_wait_ready(ready, 5, 2000, err, 3, stream=s)
    s.synchronize()
    assert int(err) == 0
    # nothing raises epoch 6: the bounded wait must give up and report slot 3
    L.lsk_wait_ready(ready, 6, 100, err, 3)
    torch.cuda.synchronize()
    assert int(err) == 1 | (3 << 8)


# ------------------------------------------------------------------ GEMM epilogues
SHAPES = [(300, 520, 200), (128, 256, 64), (1, 8, 8), (513, 264, 136), (1000, 1032, 1000)]


def _gemm_ref(epi, a, b, bias, r, b2_off, N):
    if epi == L.LSK_EPI_SWIGLU:
        return F.silu(a @ b[:N].T) * (a @ b[b2_off:b2_off + N].T)
    acc = a @ b[:N].T
    if epi == L.LSK_EPI_BIAS_GELU:
        return F.gelu(acc + bias)
    if epi == L.LSK_EPI_BIAS_RESID:
        return acc + bias + r
    if epi == L.LSK_EPI_RESID:
        return acc + r
    return acc


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("epi", [L.LSK_EPI_STORE, L.LSK_EPI_BIAS_GELU, L.LSK_EPI_BIAS_RESID,
                                 L.LSK_EPI_SWIGLU, L.LSK_EPI_RESID])
def test_gemm_epilogues_vs_oracle(M, N, K, epi):
    b_rows = 2 * N + 16 if epi == L.LSK_EPI_SWIGLU else N
    b2 = N + 16 if epi == L.LSK_EPI_SWIGLU else 0
    ab, a = rand_bf16((M, K), 1, 1.0)
    bb, b = rand_bf16((b_rows, K), 2, 1.0 / np.sqrt(K))
    biasb, bias = rand_bf16((N,), 3, 0.5)
    rb, r = rand_bf16((M, N), 4, 1.0)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    L.lsk_gemm_bf16(epi, bf16_dev(ab), bf16_dev(bb), C, M, N, K, bias=bf16_dev(biasb),
                    resid=bf16_dev(rb), b_rows=b_rows, b2_row_off=b2)
    torch.cuda.synchronize()
    _no_device_error()
    ref = _gemm_ref(epi, a, b, bias, r, b2, N)
    got = to_f64(C)
    # fp32 accumulation + one bf16 rounding: within 2^-8 of each value, plus accumulation noise
    tol = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.sqrt(K) * np.abs(ref).max()
    assert np.all(np.abs(got - ref) <= tol), (epi, np.max(np.abs(got - ref) - tol))


@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (256, 264, 72)])
@pytest.mark.parametrize("epi", [L.LSK_EPI_BIAS_RESID, L.LSK_EPI_RESID])
def test_gemm_fp32_residual_stream(M, N, K, epi):
    """Residual read in fp32, result written both as fp32 (the residual stream)
    and as its bf16 rounding (the next GEMM's operand)."""
    ab, a = rand_bf16((M, K), 31)
    bb, b = rand_bf16((N, K), 32, 1.0 / np.sqrt(K))
    biasb, bias = rand_bf16((N,), 33, 0.5)
    r = np.random.default_rng(34).standard_normal((M, N)).astype(np.float32)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    L.lsk_gemm_bf16(epi, bf16_dev(ab), bf16_dev(bb), C, M, N, K, bias=bf16_dev(biasb),
                    resid=torch.from_numpy(r).cuda(), C32=C32)
    torch.cuda.synchronize()
    _no_device_error()
    ref = a @ b.T + r.astype(np.float64) + (bias if epi == L.LSK_EPI_BIAS_RESID else 0)
    got32 = C32.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got32 - ref)) <= 1e-5 * np.sqrt(K) * np.abs(ref).max()
    # the bf16 output is exactly the rounding of the fp32 output
    assert torch.equal(C.cpu(), C32.cpu().to(torch.bfloat16))


@pytest.mark.parametrize("ctas", [1, 3, 37, 0])
def test_gemm_bit_identical_across_grid_sizes(ctas):
    M, N, K = 700, 776, 320
    ab, _ = rand_bf16((M, K), 5)
    bb, _ = rand_bf16((N, K), 6, 0.1)
    A, B = bf16_dev(ab), bf16_dev(bb)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    L.lsk_gemm_bf16(L.LSK_EPI_STORE, A, B, ref, M, N, K, max_ctas=0)
    out = torch.empty_like(ref)
    L.lsk_gemm_bf16(L.LSK_EPI_STORE, A, B, out, M, N, K, max_ctas=ctas)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


# Small GEMMs (M <= 128) with few 256-column tiles are split along K: each slice's partial tile
# is written in fp32 and a reduction adds them in slice order, then runs the epilogue. On a
# 152-SM device these take 16, 5, 16 and 2 slices.
SPLIT_SHAPES = [(128, 1024, 4096), (100, 4096, 1024), (1, 520, 2000), (77, 264, 304)]


@pytest.mark.parametrize("M,N,K", SPLIT_SHAPES)
@pytest.mark.parametrize("epi", [L.LSK_EPI_STORE, L.LSK_EPI_BIAS_GELU, L.LSK_EPI_BIAS_RESID, L.LSK_EPI_RESID])
def test_split_k_gemm_vs_oracle(M, N, K, epi):
    ab, a = rand_bf16((M, K), 41, 1.0)
    bb, b = rand_bf16((N, K), 42, 1.0 / np.sqrt(K))
    biasb, bias = rand_bf16((N,), 43, 0.5)
    r = np.random.default_rng(44).standard_normal((M, N)).astype(np.float32)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    resid = epi in (L.LSK_EPI_BIAS_RESID, L.LSK_EPI_RESID)
    A, B, Bias, R = bf16_dev(ab), bf16_dev(bb), bf16_dev(biasb), torch.from_numpy(r).cuda()
    L.lsk_gemm_bf16(epi, A, B, C, M, N, K, bias=Bias, resid=R, C32=C32 if resid else None)
    torch.cuda.synchronize()
    _no_device_error()
    ref = _gemm_ref(epi, a, b, bias, r.astype(np.float64), 0, N)
    got = to_f64(C)
    tol = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.sqrt(K) * np.abs(ref).max()
    assert np.all(np.abs(got - ref) <= tol), (epi, np.max(np.abs(got - ref) - tol))
    if resid:
        assert torch.equal(C.cpu(), C32.cpu().to(torch.bfloat16))
    # the slice count depends on the shape only: the grid a call gets does not change a bit
    for ctas in (7, 37):
        out = torch.empty_like(C)
        L.lsk_gemm_bf16(epi, A, B, out, M, N, K, bias=Bias, resid=R, C32=C32 if resid else None,
                        max_ctas=ctas)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), C.view(torch.int16)), ctas


# Tile widths of the pair GEMM: on a 152-SM device these shapes (ragged M and N) take
# 256 x 160, 192, 224 and 256 tiles.
TILE_N_SHAPES = {160: (300, 520, 200), 192: (520, 4008, 200), 224: (520, 4808, 200), 256: (520, 5608, 200)}


def test_gemm_tile_widths_cover_every_width():
    got = {w: L.lsk_gemm_tile_n(L.LSK_EPI_STORE, *TILE_N_SHAPES[w][:2]) for w in TILE_N_SHAPES}
    assert all(v in (160, 192, 224, 256) for v in got.values())
    if L.lsk_num_sms() == 152:
        assert got == {w: w for w in TILE_N_SHAPES}
    assert L.lsk_gemm_tile_n(L.LSK_EPI_SWIGLU, 4096, 4096) == 128
    assert L.lsk_gemm_tile_n(L.LSK_EPI_STORE, 128, 4096) == 256   # single-CTA tiles
    assert L.lsk_gemm_tile_n(9, 4096, 4096) == 0


@pytest.mark.parametrize("width", sorted(TILE_N_SHAPES))
@pytest.mark.parametrize("epi", [L.LSK_EPI_STORE, L.LSK_EPI_BIAS_GELU, L.LSK_EPI_BIAS_RESID, L.LSK_EPI_RESID])
def test_gemm_tile_widths_vs_oracle(width, epi):
    M, N, K = TILE_N_SHAPES[width]
    ab, a = rand_bf16((M, K), 41, 1.0)
    bb, b = rand_bf16((N, K), 42, 1.0 / np.sqrt(K))
    biasb, bias = rand_bf16((N,), 43, 0.5)
    r = np.random.default_rng(44).standard_normal((M, N)).astype(np.float32)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out32 = epi in (L.LSK_EPI_BIAS_RESID, L.LSK_EPI_RESID)
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda") if out32 else None
    L.lsk_gemm_bf16(epi, bf16_dev(ab), bf16_dev(bb), C, M, N, K, bias=bf16_dev(biasb),
                    resid=torch.from_numpy(r).cuda(), C32=C32)
    torch.cuda.synchronize()
    _no_device_error()
    ref = _gemm_ref(epi, a, b, bias, r.astype(np.float64), 0, N)
    got = to_f64(C)
    tol = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.sqrt(K) * np.abs(ref).max()
    assert np.all(np.abs(got - ref) <= tol), (epi, np.max(np.abs(got - ref) - tol))
    if out32:
        got32 = C32.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(got32 - ref)) <= 1e-5 * np.sqrt(K) * np.abs(ref).max()
        assert torch.equal(C.cpu(), C32.cpu().to(torch.bfloat16))


@pytest.mark.parametrize("width", [160, 224])
@pytest.mark.parametrize("ctas", [2, 6, 38])
def test_gemm_tile_widths_bits_independent_of_grid(width, ctas):
    M, N, K = TILE_N_SHAPES[width]
    ab, _ = rand_bf16((M, K), 45)
    bb, _ = rand_bf16((N, K), 46, 0.1)
    biasb, _ = rand_bf16((N,), 47, 0.5)
    r = torch.from_numpy(np.random.default_rng(48).standard_normal((M, N)).astype(np.float32)).cuda()
    A, B, bias = bf16_dev(ab), bf16_dev(bb), bf16_dev(biasb)
    outs = []
    for mc in (0, ctas):
        C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
        L.lsk_gemm_bf16(L.LSK_EPI_BIAS_RESID, A, B, C, M, N, K, bias=bias, resid=r, C32=C32, max_ctas=mc)
        outs.append((C, C32))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int32), outs[1][1].view(torch.int32))


# Longer K with ragged M and N (several waves of k-blocks per tile, partial last tiles).
LONG_K_SHAPES = [(1000, 1032, 4096), (300, 520, 2048), (4096, 1024, 4000)]


@pytest.mark.parametrize("M,N,K", LONG_K_SHAPES)
@pytest.mark.parametrize("epi", [L.LSK_EPI_STORE, L.LSK_EPI_BIAS_GELU, L.LSK_EPI_BIAS_RESID,
                                 L.LSK_EPI_SWIGLU, L.LSK_EPI_RESID])
def test_gemm_long_k_vs_oracle(M, N, K, epi):
    test_gemm_epilogues_vs_oracle(M, N, K, epi)


@pytest.mark.parametrize("epi", [L.LSK_EPI_BIAS_RESID, L.LSK_EPI_RESID])
def test_gemm_long_k_fp32_residual_stream(epi):
    test_gemm_fp32_residual_stream(1000, 1032, 4096, epi)


@pytest.mark.parametrize("epi", [L.LSK_EPI_STORE, L.LSK_EPI_SWIGLU])
def test_gemm_long_k_bits_independent_of_grid(epi):
    """Fewer clusters take more tiles each and produce the same bits."""
    M, N, K = 1000, 1032, 4096
    b_rows = 2 * N if epi == L.LSK_EPI_SWIGLU else N
    ab, _ = rand_bf16((M, K), 41)
    bb, _ = rand_bf16((b_rows, K), 42, 1.0 / np.sqrt(K))
    A, B = bf16_dev(ab), bf16_dev(bb)
    kw = dict(b_rows=b_rows, b2_row_off=N if epi == L.LSK_EPI_SWIGLU else 0)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    L.lsk_gemm_bf16(epi, A, B, ref, M, N, K, max_ctas=0, **kw)
    for ctas in (2, 6, 38, 0):
        out = torch.full_like(ref, float("nan"))
        L.lsk_gemm_bf16(epi, A, B, out, M, N, K, max_ctas=ctas, **kw)
        torch.cuda.synchronize()
        _no_device_error()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), ctas


# Tiles about 100 k-blocks long with ragged M and N; the second shape's K ends in a
# partial k-block.
VERY_LONG_K_SHAPES = [(1000, 1032, 6400), (300, 520, 6200)]


@pytest.mark.parametrize("M,N,K", VERY_LONG_K_SHAPES)
@pytest.mark.parametrize("epi", [L.LSK_EPI_STORE, L.LSK_EPI_BIAS_GELU, L.LSK_EPI_BIAS_RESID,
                                 L.LSK_EPI_SWIGLU, L.LSK_EPI_RESID])
def test_gemm_very_long_k_vs_oracle(M, N, K, epi):
    test_gemm_epilogues_vs_oracle(M, N, K, epi)


@pytest.mark.parametrize("epi", [L.LSK_EPI_BIAS_RESID, L.LSK_EPI_RESID])
def test_gemm_very_long_k_fp32_residual_stream(epi):
    test_gemm_fp32_residual_stream(1000, 1032, 6400, epi)


@pytest.mark.parametrize("epi", [L.LSK_EPI_STORE, L.LSK_EPI_SWIGLU, L.LSK_EPI_BIAS_RESID])
def test_gemm_very_long_k_bits_independent_of_grid(epi):
    """Fewer clusters take more tiles each and produce the same bits (residual epilogue
    included)."""
    M, N, K = 1000, 1032, 6400
    b_rows = 2 * N if epi == L.LSK_EPI_SWIGLU else N
    ab, _ = rand_bf16((M, K), 51)
    bb, _ = rand_bf16((b_rows, K), 52, 1.0 / np.sqrt(K))
    biasb, _ = rand_bf16((N,), 53, 0.5)
    rb, _ = rand_bf16((M, N), 54, 1.0)
    A, B = bf16_dev(ab), bf16_dev(bb)
    kw = dict(b_rows=b_rows, b2_row_off=N if epi == L.LSK_EPI_SWIGLU else 0, bias=bf16_dev(biasb),
              resid=bf16_dev(rb))
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    L.lsk_gemm_bf16(epi, A, B, ref, M, N, K, max_ctas=0, **kw)
    for ctas in (2, 6, 38, 0):
        out = torch.full_like(ref, float("nan"))
        L.lsk_gemm_bf16(epi, A, B, out, M, N, K, max_ctas=ctas, **kw)
        torch.cuda.synchronize()
        _no_device_error()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), ctas


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 1024), (4096, 1024, 4096)])
def test_gemm_full_size_sampled_rows(M, N, K):
    """The stack's own GEMM shapes in the launch configuration ls_run uses,
    checked on sampled rows against the oracle."""
    ab, a = rand_bf16((M, K), 7)
    bb, b = rand_bf16((N, K), 8, 1.0 / np.sqrt(K))
    biasb, bias = rand_bf16((N,), 9, 0.3)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    L.lsk_gemm_bf16(L.LSK_EPI_BIAS_GELU, bf16_dev(ab), bf16_dev(bb), C, M, N, K, bias=bf16_dev(biasb))
    torch.cuda.synchronize()
    _no_device_error()
    rows = np.random.default_rng(0).choice(M, 64, replace=False)
    ref = F.gelu(a[rows] @ b.T + bias)
    got = to_f64(C)[rows]
    assert rel_err(got, ref) <= 4e-3


# ------------------------------------------------------------------ grouped (expert) GEMM
def _groups(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


@pytest.mark.parametrize("sizes", [[130, 0, 5, 300, 128, 1], [0, 0, 64], [257] * 3, [7]])
def test_grouped_swiglu_and_scaled_down(sizes):
    G = len(sizes)
    H, Fh, k = 256, 192, 2
    rows = int(sum(sizes))
    bounds = _groups(sizes)
    xb, x = rand_bf16((rows, H), 11)
    # per expert: G [Fh, H], U [Fh, H] stacked as rows; D [H, Fh] in its own view
    gub, gu = rand_bf16((G * 2 * Fh, H), 12, 1 / np.sqrt(H))
    db, d = rand_bf16((G * H, Fh), 13, 1 / np.sqrt(Fh))
    hs = torch.zeros((max(rows, 1), Fh), dtype=torch.bfloat16, device="cuda")
    L.lsk_gemm_grouped_bf16(L.LSK_EPI_SWIGLU, bf16_dev(xb), bf16_dev(gub), G * 2 * Fh, 0, 2 * Fh, Fh,
                            torch.from_numpy(bounds).cuda(), G, hs, rows, Fh, H)
    torch.cuda.synchronize()
    _no_device_error()
    href = np.zeros((rows, Fh))
    for g in range(G):
        r0, r1 = bounds[g], bounds[g + 1]
        gg = gu[g * 2 * Fh:g * 2 * Fh + Fh]
        uu = gu[g * 2 * Fh + Fh:(g + 1) * 2 * Fh]
        href[r0:r1] = F.silu(x[r0:r1] @ gg.T) * (x[r0:r1] @ uu.T)
    got_h = to_f64(hs)[:rows]
    if rows:
        assert rel_err(got_h, href) <= 4e-3
    # down projection, scaled and scattered through a row table
    perm = np.random.default_rng(3).permutation(rows).astype(np.int32)
    w = np.random.default_rng(4).random(max(rows, 1)).astype(np.float32)
    Y = torch.full((max(rows, 1), H), float("nan"), dtype=torch.float32, device="cuda")
    L.lsk_gemm_grouped_bf16(L.LSK_EPI_SCALE_F32, hs, bf16_dev(db), G * H, 0, H, 0,
                            torch.from_numpy(bounds).cuda(), G, Y, rows, H, Fh,
                            row_table=torch.from_numpy(perm).cuda(), row_weight=torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    _no_device_error()
    if rows:
        hq = to_f64(hs)[:rows]   # the GPU's own bf16 H isolates the down GEMM
        yref = np.zeros((rows, H))
        for g in range(G):
            r0, r1 = bounds[g], bounds[g + 1]
            yref[perm[r0:r1]] = w[perm[r0:r1], None] * (hq[r0:r1] @ d[g * H:(g + 1) * H].T)
        assert rel_err(Y.cpu().numpy()[:rows].astype(np.float64), yref) <= 1e-5


# ------------------------------------------------------------------ fp32 linear + GELU
@pytest.mark.parametrize("T,H,Fo", [(8, 256, 256), (1, 32, 8), (37, 100, 260)])
def test_linear_gelu_f32(T, H, Fo):
    r = np.random.default_rng(T)
    x = r.standard_normal((T, H)).astype(np.float32)
    w = (r.standard_normal((Fo, H)) / np.sqrt(H)).astype(np.float32)
    b = (r.standard_normal(Fo) / np.sqrt(H)).astype(np.float32)
    y = torch.empty((T, Fo), dtype=torch.float32, device="cuda")
    L.lsk_linear_gelu_f32(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(),
                          torch.from_numpy(b).cuda(), y, T, H, Fo)
    torch.cuda.synchronize()
    ref = F.linear_gelu(x.astype(np.float64), w.astype(np.float64), b.astype(np.float64))
    assert np.max(np.abs(y.cpu().numpy() - ref)) <= 1e-5


# ------------------------------------------------------------------ MoE routing
@pytest.mark.parametrize("T,E,k", [(2048, 128, 8), (33, 16, 3), (5, 8, 8), (1, 256, 1)])
def test_route_and_group_exact(T, E, k):
    nl = 2
    r = np.random.default_rng(E + k)
    lg = r.standard_normal((nl, T, E)).astype(np.float32)
    lg[0, 0, :] = 0.25                  # an all-tied row
    if T > 1:
        lg[1, 1, ::3] = 2.0             # many ties at the top
    sel = torch.empty((nl, T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((nl, T, k), dtype=torch.float32, device="cuda")
    L.lsk_moe_route(torch.from_numpy(lg).cuda(), nl, T, E, k, sel, w)
    table = torch.empty((nl, T * k), dtype=torch.int32, device="cuda")
    bounds = torch.empty((nl, E + 1), dtype=torch.int32, device="cuda")
    used = torch.empty((nl, E), dtype=torch.uint8, device="cuda")
    L.lsk_moe_group(sel, nl, T, E, k, table, bounds, used)
    torch.cuda.synchronize()
    for l in range(nl):
        rs, rw = F.route_topk(lg[l], k)
        np.testing.assert_array_equal(sel[l].cpu().numpy(), rs)
        np.testing.assert_allclose(w[l].cpu().numpy(), rw, rtol=0, atol=2e-6)
        rt, rb = F.group_by_expert(rs, E)
        np.testing.assert_array_equal(table[l].cpu().numpy(), rt)
        np.testing.assert_array_equal(bounds[l].cpu().numpy(), rb)
        np.testing.assert_array_equal(used[l].cpu().numpy(), (np.diff(rb) > 0).astype(np.uint8))


def test_gather_and_combine():
    T, k, H = 77, 3, 64
    xb, x = rand_bf16((T, H), 21)
    table = np.random.default_rng(2).permutation(T * k).astype(np.int32)
    xs = torch.empty((T * k, H), dtype=torch.bfloat16, device="cuda")
    L.lsk_moe_gather(bf16_dev(xb), torch.from_numpy(table).cuda(), T * k, k, H, xs)
    y = np.random.default_rng(3).standard_normal((T * k, H)).astype(np.float32)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    L.lsk_moe_combine(bf16_dev(xb), torch.from_numpy(y).cuda(), T, k, H, out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_f64(xs), x[table // k])
    ref = x + y.astype(np.float64).reshape(T, k, H).sum(1)
    assert np.all(np.abs(to_f64(out) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)
    # fp32 residual in, fp32 residual out
    xf = np.random.default_rng(5).standard_normal((T, H)).astype(np.float32)
    out32 = torch.empty((T, H), dtype=torch.float32, device="cuda")
    L.lsk_moe_combine(torch.from_numpy(xf).cuda(), torch.from_numpy(y).cuda(), T, k, H, out, out32=out32)
    torch.cuda.synchronize()
    ref32 = xf.astype(np.float64) + y.astype(np.float64).reshape(T, k, H).sum(1)
    assert np.max(np.abs(out32.cpu().numpy() - ref32)) <= 1e-5
    assert torch.equal(out.cpu(), out32.cpu().to(torch.bfloat16))
