"""GPU: the ExpCast device function (its reference form, and the per-row form
the 8-bit attention kernel runs) and the format encoders are bit-exact with the
oracle; every tcgen05 operand layout the kernels use multiplies correctly."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V():
    from bit_attention_video_gb300 import vca
    vca.lib()
    return vca


def test_expcast_device_function_bit_exact(V, orc):
    rng = np.random.default_rng(11)
    n = 1 << 20
    a = rng.uniform(0.01, 3.0, n).astype(np.float32)
    acc = rng.uniform(-400, 400, n).astype(np.float32)
    M = (a * np.float32(400) * rng.uniform(0.5, 1.0, n).astype(np.float32)).astype(np.float32)
    b = (np.float32(119.65) - M).astype(np.float32)
    # exact rounding ties of fma(a, acc, b): a = 1, acc = k + 0.5 - b
    k = rng.integers(-5, 125, 4096)
    a[:4096] = 1.0
    b[:4096] = np.float32(0.0)
    acc[:4096] = (k + 0.5).astype(np.float32)
    acc[4096:4099] = [np.nan, -np.inf, np.inf]
    ref = orc.expcast_f32(acc, a, b)
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    V.debug_expcast(torch.from_numpy(acc).cuda(), torch.from_numpy(a).cuda(),
                    torch.from_numpy(b).cuda(), out)
    got = out.cpu().numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}: {got[bad[:5]]} vs {ref[bad[:5]]}"


def _expcast_rows_inputs():
    """Rows of 128 raw scores with the kernel's per-row scale a and previous
    running maximum M: random rows (first block, no rise, rise), exact
    rounding ties of the FMA, both clip ends, masked tails, NaN scores, |M|
    on both sides of 2^20 (where the kernel switches between its two forms)
    and beyond, and tiny a."""
    rng = np.random.default_rng(31)
    R = 8192
    s = np.zeros((R, 128), np.float32)
    a = np.ones(R, np.float32)
    M = np.full(R, -np.inf, np.float32)
    valid = np.full(R, 128, np.int32)
    # random rows: a * s spans tens to hundreds below the maximum
    n = 4096
    a[:n] = (10.0 ** rng.uniform(-4, 0.5, n)).astype(np.float32)
    sig = rng.uniform(1, 60, n) / a[:n]
    s[:n] = (rng.standard_normal((n, 128)) * sig[:, None]).astype(np.float32)
    am = (a[:n] * s[:n].max(1)).astype(np.float32)
    kind = rng.integers(0, 3, n)
    M[:n] = np.where(kind == 0, -np.inf, np.where(kind == 1, am + rng.uniform(0, 50, n),
                                                    am - rng.uniform(0, 50, n))).astype(np.float32)
    # exact ties: b = 119.65f - M = 100 exactly, a s = t - 100 with t = k + 1/2
    r0, r1 = 4096, 4608
    M[r0:r1] = np.float32(np.float32(119.65) - np.float32(100))
    t = rng.integers(-3, 120, (r1 - r0, 128)) + 0.5
    a[r0:r1] = np.where(np.arange(r1 - r0) % 2 == 0, 1.0, 0.5).astype(np.float32)
    s[r0:r1] = ((t - 100) / a[r0:r1, None]).astype(np.float32)
    # both clip ends: t in (-1, 1) and the row maximum at 119.65
    r0, r1 = 4608, 4864
    M[r0:r1] = np.float32(np.float32(119.65) - np.float32(100))
    s[r0:r1] = rng.uniform(-101, -99, (r1 - r0, 128)).astype(np.float32)
    s[r0:r1, 0] = M[r0:r1]
    # masked tails and NaN scores
    r0, r1 = 4864, 5376
    s[r0:r1] = (rng.standard_normal((r1 - r0, 128)) * 30).astype(np.float32)
    valid[r0:r1] = rng.integers(1, 128, r1 - r0)
    s[r0 + 1::7, 5] = np.nan
    M[r0:r1:3] = np.float32(5.0)
    # |M| around 2^20 and beyond (a s within 200 of M)
    r0, r1 = 5376, 6400
    base = np.array([2 ** 20 - 1, 2 ** 20 - 0.5, 2 ** 20, 2 ** 20 + 1, 2 ** 21, 2 ** 23, 2 ** 24 + 2,
                     3 * 2 ** 24, 2 ** 30, -(2 ** 20) + 1, -(2 ** 20), -(2 ** 20) - 8, -(2 ** 24)],
                    np.float64)
    pick = base[rng.integers(0, base.size, r1 - r0)]
    a[r0:r1] = rng.choice(np.array([1.0, 3.0, 0.7, 0.125], np.float32), r1 - r0)
    s[r0:r1] = ((pick[:, None] - rng.uniform(0, 200, (r1 - r0, 128))) / a[r0:r1, None]) \
        .astype(np.float32)
    s[r0:r1, 7] = (pick / a[r0:r1]).astype(np.float32)
    M[r0:r1] = np.where(rng.integers(0, 2, r1 - r0) == 0, -np.inf, pick).astype(np.float32)
    # tiny a (scores near the fp32 maximum)
    r0, r1 = 6400, 6656
    a[r0:r1] = rng.choice(np.array([2.0 ** -121, 2.0 ** -120, 2.0 ** -119, 2.0 ** -118],
                                   np.float32), r1 - r0)
    s[r0:r1] = (rng.uniform(-100, 0, (r1 - r0, 128)) / a[r0:r1, None]).astype(np.float32)
    # the rest: ordinary rows with small scales
    r0 = 6656
    a[r0:] = np.float32(0.05)
    s[r0:] = (rng.standard_normal((R - r0, 128)) * 400).astype(np.float32)
    return s, a, M, valid


def test_expcast_kernel_form_bit_exact(V, orc):
    """The softmax step the 8-bit attention kernel runs (paper §3.3 Eq 7 with
    the running maximum of Eq 1): the paired FMA, the multiply by 2^-149 that
    rounds onto the subnormal grid and the saturating byte pack where that is
    exact, the single-FMA form elsewhere (NaN rows, |M| >= 2^20), byte for
    byte against the oracle's single-FMA fp32 form, on 2^20 scores."""
    s, a, M, valid = _expcast_rows_inputs()
    R = s.shape[0]
    codes = torch.empty((R, 128), dtype=torch.uint8, device="cuda")
    Mn = torch.empty(R, dtype=torch.float32, device="cuda")
    V.debug_expcast_rows(torch.from_numpy(s).cuda(), torch.from_numpy(a).cuda(),
                         torch.from_numpy(M).cuda(), torch.from_numpy(valid).cuda(), codes, Mn)
    got, got_mn = codes.cpu().numpy(), Mn.cpu().numpy()
    # the running maximum and the bytes the oracle gives for it
    sm = s.copy()
    sm[np.arange(128)[None, :] >= valid[:, None]] = -np.inf
    with np.errstate(invalid="ignore", over="ignore"):
        mn = np.fmax(M, (a * np.nanmax(sm, axis=1)).astype(np.float32))
        b = (np.float32(119.65) - mn).astype(np.float32)
    assert np.array_equal(got_mn, mn), f"running max differs in {np.sum(got_mn != mn)} rows"
    ref = orc.expcast_f32(sm.ravel(), np.repeat(a, 128), np.repeat(b, 128)).reshape(R, 128)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, (f"{len(bad)} bytes differ, first rows {bad[:5, 0]}: "
                           f"{got[tuple(bad[:5].T)]} vs {ref[tuple(bad[:5].T)]}")
    # the inputs reach what they are meant to: ties, both clips, both forms
    assert np.sum(ref == 120) >= R // 2 and np.sum(ref == 0) > 10000
    big = np.abs(mn) >= 2 ** 20
    assert 100 < np.sum(big) < R - 100


def test_encoders_bit_exact(V, orc):
    # every 40503rd bit pattern (~106k), random values, every E4M3 / E2M1
    # midpoint and its two float neighbours
    pats = np.arange(0, 1 << 32, 40503, dtype=np.uint64).astype(np.uint32)
    rng = np.random.default_rng(12)
    vals = [pats.view(np.float32),
            rng.standard_normal(1 << 20).astype(np.float32) * np.float32(50),
            rng.standard_normal(1 << 18).astype(np.float32) * np.float32(0.01)]
    e4 = orc.e4m3_decode(np.arange(127))
    e2 = orc.e2m1_decode(np.arange(8))
    for grid in (e4, e2):
        mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
        for m in (mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))):
            vals += [m, -m]
    x = np.concatenate(vals).astype(np.float32)
    x = x[~np.isnan(x)]
    o4 = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    o2 = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    V.debug_encode(torch.from_numpy(x).cuda(), o4, o2)
    g4, g2 = o4.cpu().numpy(), o2.cpu().numpy()
    r4 = orc.e4m3_encode_array(x)
    r2 = orc.e2m1_encode_array(x)
    assert np.array_equal(g4, r4), f"e4m3: {np.sum(g4 != r4)} mismatches at {x[g4 != r4][:5]}"
    assert np.array_equal(g2, r2), f"e2m1: {np.sum(g2 != r2)} mismatches at {x[g2 != r2][:5]}"


def _e4m3_small(rng, shape):
    # exactly representable small values so products and sums are exact in fp32
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, -0.5, -1, -2, -3, 0.25, -0.25], np.float32)
    return vals[rng.integers(0, vals.size, shape)]


def _run_mma(V, mode, a, b):
    d = torch.zeros(128, 128, dtype=torch.float32, device="cuda")
    V.debug_mma(mode, a.cuda(), b.cuda(), d)
    torch.cuda.synchronize()
    return d.cpu().numpy()


@pytest.mark.parametrize("mode,K,kind", [(0, 128, "fp8"), (1, 128, "bf16"), (2, 64, "bf16"),
                                         (3, 16, "bf16"), (4, 128, "bf16"), (5, 128, "fp8")])
def test_mma_layouts(V, mode, K, kind):
    rng = np.random.default_rng(100 + mode)
    A = _e4m3_small(rng, (128, K))
    Bm = _e4m3_small(rng, (128, K))
    if kind == "fp8":
        ta = torch.from_numpy(A).to(torch.float8_e4m3fn).view(torch.uint8)
        tb = torch.from_numpy(Bm).to(torch.float8_e4m3fn).view(torch.uint8)
    else:
        ta = torch.from_numpy(A).to(torch.bfloat16)
        tb = torch.from_numpy(Bm).to(torch.bfloat16)
    got = _run_mma(V, mode, ta, tb)
    ref = A.astype(np.float64) @ Bm.astype(np.float64).T
    if not np.array_equal(got, ref):
        diag = []
        if mode in (4, 5):  # diagnose the packing order of the TMEM operand
            g = 2 if mode == 4 else 4
            Ap = A.reshape(128, -1, g)[:, :, ::-1].reshape(128, K)
            diag.append(f"reversed packing matches: {np.array_equal(got, Ap @ Bm.T)}")
        if mode == 2:
            diag.append(f"B^T product matches: {np.array_equal(got, A @ Bm.reshape(K, 128))}")
        pytest.fail(f"mode {mode}: max |err| {np.abs(got - ref).max()}, "
                    f"{np.sum(got != ref)} mismatches; {'; '.join(diag)}")


def test_mma_mixed_kinds_one_accumulator(V):
    rng = np.random.default_rng(7)
    A8, B8 = _e4m3_small(rng, (128, 128)), _e4m3_small(rng, (128, 128))
    A16, B16 = _e4m3_small(rng, (128, 16)), _e4m3_small(rng, (128, 16))
    ta = torch.cat([torch.from_numpy(A8).to(torch.float8_e4m3fn).view(torch.uint8).ravel(),
                    torch.from_numpy(A16).to(torch.bfloat16).view(torch.uint8).ravel()])
    tb = torch.cat([torch.from_numpy(B8).to(torch.float8_e4m3fn).view(torch.uint8).ravel(),
                    torch.from_numpy(B16).to(torch.bfloat16).view(torch.uint8).ravel()])
    got = _run_mma(V, 6, ta, tb)
    ref = A8.astype(np.float64) @ B8.T + A16.astype(np.float64) @ B16.T
    assert np.array_equal(got, ref)


def _nvfp4_operand(rng, pow2_scales):
    """[128][64] packed E2M1 bytes (element 2i in the low nibble) followed by
    [128][8] UE4M3 scales; returns the bytes and the decoded [128][128] matrix."""
    from oracle import e2m1_decode, e4m3_decode
    codes = rng.integers(0, 16, (128, 128)).astype(np.uint8)
    if pow2_scales:
        sc = np.array([0x28, 0x30, 0x38, 0x40, 0x48], np.uint8)[rng.integers(0, 5, (128, 8))]
    else:
        sc = rng.integers(0x20, 0x50, (128, 8)).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    val = e2m1_decode(codes).reshape(128, 128) * np.repeat(e4m3_decode(sc).reshape(128, 8), 16, 1)
    raw = np.concatenate([packed.ravel(), sc.ravel()])
    return torch.from_numpy(raw), val


@pytest.mark.parametrize("pow2_scales", [True, False])
def test_mma_nvfp4_block_scaled(V, pow2_scales):
    """kind::mxf4nvf4 with UE4M3 scales per 16 elements: the product of the
    decoded operands.  With power-of-two scales every partial sum is exact in
    fp32; with general scales the tensor core may round its partial sums."""
    rng = np.random.default_rng(70 + pow2_scales)
    ta, A = _nvfp4_operand(rng, pow2_scales)
    tb, Bm = _nvfp4_operand(rng, pow2_scales)
    got = _run_mma(V, 7, ta, tb)
    ref = A @ Bm.T
    tol = (1e-6 if pow2_scales else 1e-5) * np.abs(ref).max()
    err = np.abs(got - ref)
    assert err.max() <= tol, f"max |err| {err.max()} (tol {tol}), {np.sum(err > tol)} mismatches"
