"""GPU grouped GEMMs (forward, dgrad, wgrad) vs the CPU oracle's fp64 GEMM over its own
quantization of the same bf16 inputs: max|gpu - oracle| <= 2e-2 * rms(oracle)."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import COL_B, ROW_B, TOL, bits, check_dev_err, dev, from_bits, np_, offsets, rel_err  # noqa: F401

pytestmark = pytest.mark.gpu


def _rand(shape, seed, std=1.0):
    return synth.randn_bf16(shape, synth.generator(seed), std=std)


def _fwd_gpu(dev, xp, w, off, poff, E, N, K):
    R = xp.shape[0]
    err = mx.new_dev_err(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    qa = mx.quantize_alloc(xp.to(dev), mx.MX_ROWWISE, offd, poffd, dev_err=err)
    qb = mx.quantize_alloc(w.reshape(E * N, K).to(dev), ROW_B, dev_err=err)
    C = torch.full((max(R, 1), N), float("nan"), dtype=torch.bfloat16, device=dev)
    mx.grouped_gemm_mxfp8_fwd(qa["q_row"], qa["sf_row"], qb["q_row"], qb["sf_row"], offd, poffd, E, R, N, K, C, err)
    check_dev_err(err)
    return C.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("counts,N,K", [
    ([512], 256, 256),
    ([0, 37, 128, 300, 1], 384, 384),
    ([129, 0, 0, 255, 64], 128, 1024),
    ([1000, 3, 260], 512, 512),
])
def test_fwd_ragged_groups(dev, counts, N, K):
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    xp = _rand((R, K), R + N + K)
    w = _rand((E, N, K), R * 3 + 1)
    got = _fwd_gpu(dev, xp, w, off, poff, E, N, K)
    oq, osf = oracle.quantize_rowwise(bits(xp))
    wq, wsf = oracle.quantize_rowwise(bits(w).reshape(E * N, K))
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        ref = oracle.gemm_nt(oq[r0:r1], osf[r0:r1], wq[e * N:(e + 1) * N], wsf[e * N:(e + 1) * N])
        err = rel_err(got[r0:r1], ref)
        assert err <= TOL, "expert %d: max err %.3g x rms" % (e, err)


def test_fwd_structured_scales(dev):
    # Diagnostic case: A and B hold +-1 / +-2 with distinct power-of-two scales per
    # (row, K block), so a misplaced scale byte would change an output by a power of
    # two.  Outputs can cancel far below their terms here, so each output is held to
    # a bound set by its own terms: bf16 rounding of the result (2^-8 |ref|) plus
    # fp32 accumulation error (2^-20 sum_k |a_k b_k|).
    E, N, K = 2, 256, 256
    counts = [130, 126]
    off, poff = offsets(counts)
    R = int(off[-1])

    def blocky(rows, cols, seed):
        r = np.random.default_rng(seed)
        mag = r.choice([1.0, 2.0], size=(rows, cols)) * r.choice([-1.0, 1.0], size=(rows, cols))
        sc = np.exp2(r.integers(-6, 7, size=(rows, cols // 32)).repeat(32, axis=1))
        return torch.from_numpy((mag * sc).astype(np.float32)).to(torch.bfloat16)
    xp = blocky(R, K, 1)
    w = blocky(E * N, K, 2).reshape(E, N, K)
    got = _fwd_gpu(dev, xp, w, off, poff, E, N, K)
    oq, osf = oracle.quantize_rowwise(bits(xp))
    wq, wsf = oracle.quantize_rowwise(bits(w).reshape(E * N, K))
    worst = 0.0
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        bq, bs = wq[e * N:(e + 1) * N], wsf[e * N:(e + 1) * N]
        ref = oracle.gemm_nt(oq[r0:r1], osf[r0:r1], bq, bs)
        mag = oracle.gemm_nt(oq[r0:r1] & 0x7F, osf[r0:r1], bq & 0x7F, bs)   # sum_k |a_k b_k|
        bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -20 * mag
        ratio = np.abs(got[r0:r1] - ref) / bound
        worst = max(worst, float(ratio.max()))
        bad = ratio > 1.0
        assert not bad.any(), "expert %d: %d bad outputs, rows %s cols %s, worst %.3g x bound" % (
            e, bad.sum(), np.unique(np.nonzero(bad)[0])[:16], np.unique(np.nonzero(bad)[1])[:16], ratio.max())
    print("structured-scales worst error / bound = %.3g" % worst)


def test_fwd_through_permute_tiny_config(dev):
    d = synth.tiny()
    T, K, E, N, k = d["T"], d["K"], d["E"], d["N"], d["k"]
    err = mx.new_dev_err(dev)
    qx = mx.quantize_alloc(d["x"].to(dev), mx.MX_ROWWISE, dev_err=err)
    qw = mx.quantize_alloc(d["w"].reshape(E * N, K).to(dev), ROW_B, dev_err=err)
    pm = mx.permute_alloc(d["ids"].to(dev), E, qx["q_row"], qx["sf_row"], dev_err=err)
    R = T * k
    C = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
    mx.grouped_gemm_mxfp8_fwd(pm["q"], pm["sf"], qw["q_row"], qw["sf_row"], pm["off"], pm["poff"], E, R, N, K, C, err)
    check_dev_err(err)
    got = C.float().cpu().numpy().astype(np.float64)
    p = oracle.permute(d["ids"].numpy(), E)
    oq, osf = oracle.quantize_rowwise(bits(d["x"]))
    wq, wsf = oracle.quantize_rowwise(bits(d["w"]).reshape(E * N, K))
    for e in range(E):
        r0, r1 = int(p["off"][e]), int(p["off"][e + 1])
        rows = p["src_row"][r0:r1]
        ref = oracle.gemm_nt(oq[rows], osf[rows], wq[e * N:(e + 1) * N], wsf[e * N:(e + 1) * N])
        assert rel_err(got[r0:r1], ref) <= TOL


@pytest.mark.parametrize("counts,N,K", [([0, 37, 128, 300, 1], 256, 384), ([200, 0, 129], 384, 128)])
def test_dgrad_ragged_groups(dev, counts, N, K):
    # forward weight W_e is [K x N] (y = x W_e^T); dX = dY W_e contracts over K
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    dy = _rand((R, K), 5 + R, std=1e-2)
    w = _rand((E * K, N), 6 + R)
    err = mx.new_dev_err(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    qa = mx.quantize_alloc(dy.to(dev), mx.MX_ROWWISE, offd, poffd, dev_err=err)
    woff = torch.arange(0, (E + 1) * K, K, dtype=torch.int32, device=dev)
    qw = mx.quantize_alloc(w.to(dev), COL_B, woff, woff, dev_err=err, ld_col=E * K)
    dX = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device=dev)
    mx.grouped_gemm_mxfp8_dgrad(qa["q_row"], qa["sf_row"], qw["q_col"], qw["sf_col"], offd, poffd, E, R, N, K, dX, err)
    check_dev_err(err)
    got = dX.float().cpu().numpy().astype(np.float64)
    oq, osf = oracle.quantize_rowwise(bits(dy))
    wo = np.arange(0, (E + 1) * K, K, dtype=np.int32)
    cq, csf = oracle.quantize_colwise_seg(bits(w), wo, wo, E * K)
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        ref = oracle.gemm_nt(oq[r0:r1], osf[r0:r1], cq[:, e * K:(e + 1) * K], csf[:, e * K // 32:(e + 1) * K // 32])
        err_e = rel_err(got[r0:r1], ref)
        assert err_e <= TOL, "expert %d: max err %.3g x rms" % (e, err_e)


@pytest.mark.parametrize("counts,N,K", [([0, 37, 128, 300, 1], 256, 384), ([500, 0, 129], 128, 256)])
def test_wgrad_ragged_groups(dev, counts, N, K):
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    dy = _rand((R, N), 8 + R, std=1e-2)
    xp = _rand((R, K), 9 + R)
    err = mx.new_dev_err(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    qd = mx.quantize_alloc(dy.to(dev), mx.MX_COLWISE, offd, poffd, dev_err=err)
    qx = mx.quantize_alloc(xp.to(dev), COL_B, offd, poffd, dev_err=err)
    ld = qd["ld_col"]
    dW = torch.full((E, N, K), float("nan"), dtype=torch.float32, device=dev)
    mx.grouped_gemm_mxfp8_wgrad(qd["q_col"], qd["sf_col"], qx["q_col"], qx["sf_col"], offd, poffd, E, N, K, ld, dW, err)
    check_dev_err(err)
    got = dW.cpu().numpy().astype(np.float64)
    dq, dsf = oracle.quantize_colwise_seg(bits(dy), off, poff, ld)
    xq, xsf = oracle.quantize_colwise_seg(bits(xp), off, poff, ld)
    for e in range(E):
        p0, p1 = int(poff[e]), int(poff[e + 1])
        if p1 == p0:
            assert np.all(got[e] == 0.0), "empty expert %d must get a zero gradient" % e
            continue
        ref = oracle.gemm_nt(dq[:, p0:p1], dsf[:, p0 // 32:p1 // 32], xq[:, p0:p1], xsf[:, p0 // 32:p1 // 32])
        err_e = rel_err(got[e], ref)
        assert err_e <= TOL, "expert %d: max err %.3g x rms" % (e, err_e)


def _run_passes(dev, xp, w, dy, off, poff, E, N, K, flags=0, ctas_per_mma=0, cluster_pairs=0):
    """Forward C = x W_e^T, dgrad dX = dY W_e and wgrad dW_e = dY_e^T x_e through the internal
    test entry (tile shape and B-scale layout chosen per call).  Returns (C, dX, dW, ld)."""
    R = xp.shape[0]
    x4 = not (flags & mx.MX_GEMM_B_SCALES_X1)
    row_b = ROW_B if x4 else mx.MX_ROWWISE
    col_b = COL_B if x4 else mx.MX_COLWISE
    err = mx.new_dev_err(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    qa = mx.quantize_alloc(xp.to(dev), mx.MX_ROWWISE, offd, poffd, dev_err=err)
    qb = mx.quantize_alloc(w.reshape(E * N, K).to(dev), row_b, dev_err=err)
    C = torch.full((max(R, 1), N), float("nan"), dtype=torch.bfloat16, device=dev)
    run = lambda *a: mx.testing_grouped_gemm(*a, err, flags=flags, ctas_per_mma=ctas_per_mma,
                                             cluster_pairs=cluster_pairs)
    assert run(mx.MX_TESTING_FWD, qa["q_row"], qa["sf_row"], qb["q_row"], qb["sf_row"], offd, poffd, E, R, N, K, 0,
               C) == 0
    qd = mx.quantize_alloc(dy.to(dev), mx.MX_ROWWISE | mx.MX_COLWISE, offd, poffd, dev_err=err)
    woff = torch.arange(0, (E + 1) * N, N, dtype=torch.int32, device=dev)
    qw = mx.quantize_alloc(w.reshape(E * N, K).to(dev), col_b, woff, woff, dev_err=err, ld_col=E * N)
    dX = torch.full((max(R, 1), K), float("nan"), dtype=torch.bfloat16, device=dev)
    assert run(mx.MX_TESTING_DGRAD, qd["q_row"], qd["sf_row"], qw["q_col"], qw["sf_col"], offd, poffd, E, R, K, N, 0,
               dX) == 0
    qx = mx.quantize_alloc(xp.to(dev), col_b, offd, poffd, dev_err=err)
    dW = torch.full((E, N, K), float("nan"), dtype=torch.float32, device=dev)
    assert run(mx.MX_TESTING_WGRAD, qd["q_col"], qd["sf_col"], qx["q_col"], qx["sf_col"], offd, poffd, E, 0, N, K,
               qd["ld_col"], dW) == 0
    check_dev_err(err)
    return C, dX, dW, qd["ld_col"]


def _check_passes(C, dX, dW, xp, w, dy, off, poff, E, N, K, ld):
    gc = C.float().cpu().numpy().astype(np.float64)
    gdx = dX.float().cpu().numpy().astype(np.float64)
    gdw = dW.cpu().numpy().astype(np.float64)
    oq, osf = oracle.quantize_rowwise(bits(xp))
    wq, wsf = oracle.quantize_rowwise(bits(w).reshape(E * N, K))
    aq, asf = oracle.quantize_rowwise(bits(dy))
    wo = np.arange(0, (E + 1) * N, N, dtype=np.int32)
    cq, csf = oracle.quantize_colwise_seg(bits(w).reshape(E * N, K), wo, wo, E * N)
    dq, dsf = oracle.quantize_colwise_seg(bits(dy), off, poff, ld)
    xq, xsf = oracle.quantize_colwise_seg(bits(xp), off, poff, ld)
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        p0, p1 = int(poff[e]), int(poff[e + 1])
        if r1 == r0:
            assert np.all(gdw[e] == 0.0), "empty expert %d must get a zero gradient" % e
            continue
        ref = oracle.gemm_nt(oq[r0:r1], osf[r0:r1], wq[e * N:(e + 1) * N], wsf[e * N:(e + 1) * N])
        assert rel_err(gc[r0:r1], ref) <= TOL, "fwd expert %d" % e
        ref = oracle.gemm_nt(aq[r0:r1], asf[r0:r1], cq[:, e * N:(e + 1) * N], csf[:, e * N // 32:(e + 1) * N // 32])
        assert rel_err(gdx[r0:r1], ref) <= TOL, "dgrad expert %d" % e
        ref = oracle.gemm_nt(dq[:, p0:p1], dsf[:, p0 // 32:p1 // 32], xq[:, p0:p1], xsf[:, p0 // 32:p1 // 32])
        assert rel_err(gdw[e], ref) <= TOL, "wgrad expert %d" % e


@pytest.mark.parametrize("ctas", [1, 2])
@pytest.mark.parametrize("counts,N,K", [([0, 37, 128, 300, 1], 384, 384), ([1000, 3, 260], 256, 512)])
def test_tile_shapes_fwd_dgrad_wgrad(dev, counts, N, K, ctas):
    # both tile shapes on ragged groups, chosen through the internal test entry: 128 x 256
    # single-CTA tiles (cta_group::1) and 256 x 256 CTA-pair tiles (cta_group::2).  The public
    # calls pick single-CTA tiles for forward / dgrad problems this small (experts averaging
    # fewer than 512 rows), pairs at the MoE FFN sizes.
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    xp, w, dy = _rand((R, K), 11 + R), _rand((E, N, K), 12 + R), _rand((R, N), 13 + R, std=1e-2)
    C, dX, dW, ld = _run_passes(dev, xp, w, dy, off, poff, E, N, K, ctas_per_mma=ctas)
    _check_passes(C, dX, dW, xp, w, dy, off, poff, E, N, K, ld)


@pytest.mark.parametrize("ctas", [2, 1])
@pytest.mark.parametrize("counts,N,K", [([0, 37, 128, 300, 1], 384, 384), ([129, 0, 255, 64], 256, 256)])
def test_one_copy_b_scales_fwd_dgrad_wgrad(dev, counts, N, K, ctas):
    # B-operand scales in the plain one-copy layout (MX_GEMM_B_SCALES_X1): against the oracle,
    # and byte for byte the outputs of the four-copy layout (same codes, same scales, same MMAs)
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    xp, w, dy = _rand((R, K), 21 + R), _rand((E, N, K), 22 + R), _rand((R, N), 23 + R, std=1e-2)
    C, dX, dW, ld = _run_passes(dev, xp, w, dy, off, poff, E, N, K, flags=mx.MX_GEMM_B_SCALES_X1, ctas_per_mma=ctas)
    _check_passes(C, dX, dW, xp, w, dy, off, poff, E, N, K, ld)
    C4, dX4, dW4, _ = _run_passes(dev, xp, w, dy, off, poff, E, N, K, ctas_per_mma=ctas)
    assert torch.equal(C[:R].view(torch.int16), C4[:R].view(torch.int16))
    assert torch.equal(dX[:R].view(torch.int16), dX4[:R].view(torch.int16))
    assert torch.equal(dW.view(torch.int32), dW4.view(torch.int32))


@pytest.mark.parametrize("ctas", [2, 1])
@pytest.mark.parametrize("counts,N,K", [([0, 37, 128, 300, 1], 640, 384), ([600, 0, 300, 1000], 512, 256)])
def test_two_pair_clusters(dev, counts, N, K, ctas):
    # clusters sharing an operand by multicast (internal option cluster_pairs = 2): two CTA pairs on
    # the two N tiles of one M tile sharing A, with an odd N-tile count (N = 640: the second pair's
    # last tile lies past N and is not stored); or two single CTAs on two M tiles of one N tile
    # sharing B, with odd M-tile counts (the second CTA's last tile lies past the expert's rows):
    # against the oracle, and byte for byte the outputs without clusters
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    xp, w, dy = _rand((R, K), 41 + R), _rand((E, N, K), 42 + R), _rand((R, N), 43 + R, std=1e-2)
    C, dX, dW, ld = _run_passes(dev, xp, w, dy, off, poff, E, N, K, ctas_per_mma=ctas, cluster_pairs=2)
    _check_passes(C, dX, dW, xp, w, dy, off, poff, E, N, K, ld)
    C1, dX1, dW1, _ = _run_passes(dev, xp, w, dy, off, poff, E, N, K, ctas_per_mma=ctas, cluster_pairs=1)
    assert torch.equal(C[:R].view(torch.int16), C1[:R].view(torch.int16))
    assert torch.equal(dX[:R].view(torch.int16), dX1[:R].view(torch.int16))
    assert torch.equal(dW.view(torch.int32), dW1.view(torch.int32))


@pytest.mark.parametrize("ctas,cluster_pairs", [(1, 0), (1, 2), (2, 1), (2, 2)])
def test_max_experts_mostly_empty(dev, ctas, cluster_pairs):
    # E = 1024 (the largest expert count the calls take; the tile table fills its shared-memory
    # array) with 40 experts holding rows, 984 empty: forward, dgrad and wgrad against the oracle
    # per expert, empty experts' weight gradients exactly zero
    E, N, K = 1024, 128, 256
    counts = [0] * E
    rng = np.random.default_rng(1024)
    for e in sorted(rng.choice(E, 40, replace=False)):
        counts[int(e)] = int(rng.integers(1, 300))
    off, poff = offsets(counts)
    R = int(off[-1])
    xp, w, dy = _rand((R, K), 51), _rand((E, N, K), 52), _rand((R, N), 53, std=1e-2)
    C, dX, dW, ld = _run_passes(dev, xp, w, dy, off, poff, E, N, K, ctas_per_mma=ctas, cluster_pairs=cluster_pairs)
    _check_passes(C, dX, dW, xp, w, dy, off, poff, E, N, K, ld)


def test_public_ex_calls_take_one_copy_b_scales(dev):
    # the public *_ex entries with MX_GEMM_B_SCALES_X1 give the default calls' outputs
    counts, N, K = [300, 0, 129], 256, 384
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    xp, w = _rand((R, K), 31), _rand((E, N, K), 32)
    err = mx.new_dev_err(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    qa = mx.quantize_alloc(xp.to(dev), mx.MX_ROWWISE, offd, poffd, dev_err=err)
    qb1 = mx.quantize_alloc(w.reshape(E * N, K).to(dev), mx.MX_ROWWISE, dev_err=err)
    qb4 = mx.quantize_alloc(w.reshape(E * N, K).to(dev), ROW_B, dev_err=err)
    C1 = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
    C4 = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
    mx.grouped_gemm_mxfp8_fwd_ex(qa["q_row"], qa["sf_row"], qb1["q_row"], qb1["sf_row"], offd, poffd, E, R, N, K, C1,
                                 mx.MX_GEMM_B_SCALES_X1, err)
    mx.grouped_gemm_mxfp8_fwd(qa["q_row"], qa["sf_row"], qb4["q_row"], qb4["sf_row"], offd, poffd, E, R, N, K, C4, err)
    check_dev_err(err)
    assert torch.equal(C1.view(torch.int16), C4.view(torch.int16))
    with pytest.raises(mx.MxError):
        mx.grouped_gemm_mxfp8_fwd_ex(qa["q_row"], qa["sf_row"], qb1["q_row"], qb1["sf_row"], offd, poffd, E, R, N, K,
                                     C1, 4, err)


def test_dense_matches_library_mxfp8(dev):
    # An independent implementation of the same block-scaled product: the library MXFP8 GEMM
    # (torch._scaled_mm with E8M0 1x32 scales) reads the scales in the same tensor-core layout.
    # Fed the same codes and scales it must give the same bf16 outputs (observed: identical);
    # allowed: rare last-bit differences from a different fp32 accumulation order.
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch without E8M0")
    M, N, K = 640, 512, 1024
    x = _rand((M, K), 91).to(dev)
    w = _rand((N, K), 92).to(dev)
    qa = mx.quantize_alloc(x, mx.MX_ROWWISE)
    qb = mx.quantize_alloc(w, mx.MX_ROWWISE)
    qb4 = mx.quantize_alloc(w, ROW_B)
    off = torch.tensor([0, M], dtype=torch.int32, device=dev)
    C = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    err = mx.new_dev_err(dev)
    mx.grouped_gemm_mxfp8_fwd(qa["q_row"], qa["sf_row"], qb4["q_row"], qb4["sf_row"], off, off, 1, M, N, K, C, err)
    check_dev_err(err)
    try:
        lib = torch._scaled_mm(qa["q_row"].view(torch.float8_e4m3fn), qb["q_row"].view(torch.float8_e4m3fn).t(),
                               qa["sf_row"].view(torch.float8_e8m0fnu), qb["sf_row"].view(torch.float8_e8m0fnu),
                               out_dtype=torch.bfloat16)
    except (RuntimeError, TypeError, NotImplementedError) as e:
        pytest.skip("library MXFP8 GEMM unavailable: %s" % str(e)[:120])
    got, ref = C.float().cpu().numpy(), lib.float().cpu().numpy()
    diff = np.abs(got - ref)
    assert np.mean(diff != 0) <= 1e-3, "outputs differ from the library in %.3g of the elements" % np.mean(diff != 0)
    assert np.all(diff <= 2.0 ** -7 * np.abs(ref) + 1e-30)


@pytest.mark.parametrize("group", [1, 3, 8])
def test_tile_order_does_not_change_results(dev, group):
    # every tile order inside an expert (groups of M tiles, M fastest; 1 = N fastest) gives the
    # default order's bytes
    counts, N, K = [300, 0, 700, 129, 1], 768, 256
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    xp, w, dy = _rand((R, K), 41), _rand((E, N, K), 42), _rand((R, N), 43, std=1e-2)
    ref = _run_passes(dev, xp, w, dy, off, poff, E, N, K)
    for ctas in (2, 1):
        got = _run_passes_ordered(dev, xp, w, dy, off, poff, E, N, K, ctas, group)
        for a, b in zip(got[:3], ref[:3]):
            assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a[:R].view(torch.int16),
                               b.view(torch.int32) if b.dtype == torch.float32 else b[:R].view(torch.int16))


def _run_passes_ordered(dev, xp, w, dy, off, poff, E, N, K, ctas, group):
    R = xp.shape[0]
    err = mx.new_dev_err(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    qa = mx.quantize_alloc(xp.to(dev), mx.MX_ROWWISE, offd, poffd, dev_err=err)
    qb = mx.quantize_alloc(w.reshape(E * N, K).to(dev), ROW_B, dev_err=err)
    C = torch.full((max(R, 1), N), float("nan"), dtype=torch.bfloat16, device=dev)
    run = lambda *a: mx.testing_grouped_gemm(*a, err, ctas_per_mma=ctas, raster_group=group)
    assert run(mx.MX_TESTING_FWD, qa["q_row"], qa["sf_row"], qb["q_row"], qb["sf_row"], offd, poffd, E, R, N, K, 0,
               C) == 0
    qd = mx.quantize_alloc(dy.to(dev), mx.MX_ROWWISE | mx.MX_COLWISE, offd, poffd, dev_err=err)
    woff = torch.arange(0, (E + 1) * N, N, dtype=torch.int32, device=dev)
    qw = mx.quantize_alloc(w.reshape(E * N, K).to(dev), COL_B, woff, woff, dev_err=err, ld_col=E * N)
    dX = torch.full((max(R, 1), K), float("nan"), dtype=torch.bfloat16, device=dev)
    assert run(mx.MX_TESTING_DGRAD, qd["q_row"], qd["sf_row"], qw["q_col"], qw["sf_col"], offd, poffd, E, R, K, N, 0,
               dX) == 0
    qx = mx.quantize_alloc(xp.to(dev), COL_B, offd, poffd, dev_err=err)
    dW = torch.full((E, N, K), float("nan"), dtype=torch.float32, device=dev)
    assert run(mx.MX_TESTING_WGRAD, qd["q_col"], qd["sf_col"], qx["q_col"], qx["sf_col"], offd, poffd, E, 0, N, K,
               qd["ld_col"], dW) == 0
    check_dev_err(err)
    return C, dX, dW
