"""GPU quantisers (bsg_quantize through the C ABI) against the CPU oracle: bit-exact codes,
bit-exact swizzled scale buffers (padding included) and the NVFP4 global scale."""

import numpy as np
import pytest
import torch

import fp4_gemm_blackwell_gb300 as bsg
from fp4_gemm_blackwell_gb300 import synth
from oracle import formats as F
from oracle import layout as L
from oracle import quantize as Q

pytestmark = pytest.mark.gpu


def gpu_quantize(kind, x):
    rows, K = x.shape
    k = bsg.BSG_MXFP8 if kind == "mxfp8" else bsg.BSG_NVFP4
    xd = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    nb = rows * K if kind == "mxfp8" else rows * K // 2
    codes = torch.full((nb,), 0xCD, dtype=torch.uint8, device="cuda")
    sf = torch.full((bsg.bsg_sf_bytes(k, rows, K),), 0xAB, dtype=torch.uint8, device="cuda")
    gs = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    bsg.bsg_quantize(k, xd, rows, K, codes, sf, gs)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), sf.cpu().numpy(), gs.item()


def gpu_quantize_bf16(kind, bits):
    rows, K = bits.shape
    k = bsg.BSG_MXFP8 if kind == "mxfp8" else bsg.BSG_NVFP4
    xd = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    nb = rows * K if kind == "mxfp8" else rows * K // 2
    codes = torch.full((nb,), 0xCD, dtype=torch.uint8, device="cuda")
    sf = torch.full((bsg.bsg_sf_bytes(k, rows, K),), 0xAB, dtype=torch.uint8, device="cuda")
    gs = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    bsg.bsg_quantize_bf16(k, xd, rows, K, codes, sf, gs)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), sf.cpu().numpy(), gs.item()


def check(kind, x, bf16=False):
    """x: float32 values, or (bf16=True) BF16 bit patterns."""
    codes, sf, gs = gpu_quantize_bf16(kind, x) if bf16 else gpu_quantize(kind, x)
    if kind == "mxfp8":
        oc, osf = Q.quantize_mxfp8_bf16(x) if bf16 else Q.quantize_mxfp8(x)
    else:
        oc, osf, s = Q.quantize_nvfp4_bf16(x) if bf16 else Q.quantize_nvfp4(x)
        assert np.float32(gs) == s
    assert np.array_equal(codes, oc.ravel()), "codes differ at %s" % np.flatnonzero(codes != oc.ravel())[:8]
    want = L.swizzle(osf)
    assert np.array_equal(sf, want), "scales differ at %s" % np.flatnonzero(sf != want)[:8]


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("rows,K", [(1, 32), (128, 256), (200, 96), (129, 160), (256, 4096), (1000, 512)])
def test_quantiser_matches_oracle(kind, rows, K):
    gen = synth.normal if kind == "mxfp8" else synth.normal_rowscaled
    check(kind, gen(rows, K, seed=rows + K))


def test_mx_ties_extremes_and_signs():
    pos = F.E4M3_VALUES[:0x7F]
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)             # every E4M3 tie
    rows = []
    for i in range(0, len(mids), 31):
        blk = np.zeros(32, dtype=np.float32)
        blk[0] = 448.0                                                 # amax 448 -> scale 2^0
        chunk = mids[i:i + 31]
        blk[1:1 + len(chunk)] = chunk * np.where(np.arange(len(chunk)) % 2, -1, 1)
        rows.append(blk)
    special = np.zeros(32, dtype=np.float32)                          # an all-zero block
    tiny = np.full(32, 1e-41, dtype=np.float32)                       # subnormal amax
    huge = np.linspace(-3e38, 3e38, 32).astype(np.float32)
    neg_small = np.array([-1e-9] * 16 + [1.0] * 16, dtype=np.float32)  # negatives that round to -0
    x = np.stack(rows + [special, tiny, huge, neg_small])
    check("mxfp8", x)


def test_nv_closed_form_ties_and_zero_tensor():
    # s = 2688 / 2688 = 1; the block with amax 6 has scale 1, so elements are E2M1(x) directly
    row0 = np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -5.0, 0.1, 0.3, 4.4, -6.0, 1.0] * 2,
                    dtype=np.float32)
    row1 = np.zeros(32, dtype=np.float32)
    row1[0] = 2688.0
    check("nvfp4", np.stack([row0, row1]))
    check("nvfp4", np.zeros((3, 64), dtype=np.float32))


def test_full_size_operand_rows():
    # an 8192 x 8192 NVFP4 operand and an 8000-row MXFP8 operand, compared whole
    check("nvfp4", synth.normal_rowscaled(8192, 8192, seed=1))
    check("mxfp8", synth.normal(8000, 8192, seed=0))


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("rows,K", [(1, 32), (128, 256), (200, 96), (129, 160), (256, 4096), (1000, 512)])
def test_bf16_quantiser_matches_oracle(kind, rows, K):
    gen = synth.normal if kind == "mxfp8" else synth.normal_rowscaled
    check(kind, synth.as_bf16_bits(gen(rows, K, seed=rows + K)), bf16=True)


def test_bf16_ties_extremes_and_zero():
    # every E4M3 tie (four fraction bits: exact in BF16) with amax 448, a zero block, the largest
    # and smallest BF16 magnitudes; NVFP4 closed-form row and an all-zero tensor
    pos = F.E4M3_VALUES[:0x7F]
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    rows = []
    for i in range(0, len(mids), 31):
        blk = np.zeros(32, dtype=np.float32)
        blk[0] = 448.0
        chunk = mids[i:i + 31]
        blk[1:1 + len(chunk)] = chunk * np.where(np.arange(len(chunk)) % 2, -1, 1)
        rows.append(blk)
    rows.append(np.zeros(32, dtype=np.float32))
    big = np.full(32, float.fromhex("0x1.fep127"), dtype=np.float32)
    big[1::2] *= -1
    rows.append(big)
    rows.append(np.full(32, 2.0 ** -133, dtype=np.float32))
    x = np.stack(rows)
    bits = synth.as_bf16_bits(x)
    assert np.array_equal(F.decode_bf16(bits).astype(np.float32), x)     # the values survive as BF16
    check("mxfp8", bits, bf16=True)
    row0 = np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -5.0, 0.1, 0.3, 4.4, -6.0, 1.0] * 2,
                    dtype=np.float32)
    row1 = np.zeros(32, dtype=np.float32)
    row1[0] = 2688.0
    check("nvfp4", synth.as_bf16_bits(np.stack([row0, row1])), bf16=True)
    check("nvfp4", np.zeros((3, 64), dtype=np.uint16), bf16=True)


def test_bf16_full_size_operand():
    check("nvfp4", synth.as_bf16_bits(synth.normal_rowscaled(8192, 8192, seed=1)), bf16=True)
    check("mxfp8", synth.as_bf16_bits(synth.normal(8000, 8192, seed=0)), bf16=True)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_grid_stride_crosses_row_ends(kind, bf16):
    # 20000 x 1120: 35 MXFP8 or 70 NVFP4 blocks a row and more blocks than either quantiser's
    # grid has threads, so every thread visits several blocks a grid stride apart, and the stride
    # (a multiple of 256 threads) is no multiple of the blocks per row: a thread's next block
    # lies in another column of a later row.  The smaller cases give each thread one block, and
    # the 8192-wide ones a stride that keeps the column.
    gen = synth.normal if kind == "mxfp8" else synth.normal_rowscaled
    x = gen(20000, 1120, seed=7)
    check(kind, synth.as_bf16_bits(x) if bf16 else x, bf16=bf16)


def test_nv_elements_at_rounding_thresholds():
    # One element of 2688 makes s = 1, so a block whose largest magnitude is 6 v (v a UE4M3 value)
    # gets den = v exactly.  With v not a power of two, x / den and x * (1 / den) can round
    # differently; elements RN(T v) and up to 3 float32 ulps either side, for every E2M1 rounding
    # threshold T, check that the kernel's element codes are those of RN(x / den) exactly.
    thresholds = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    dens = [1.125, 1.375, 0.8125, 3.25, 0.5625, 7.0, 0.1171875, 13.0]
    blocks = []
    for v in dens:
        cand = []
        for T in thresholds:
            base = np.float32(T * v)
            lo = hi = base
            cand.append(base)
            for _ in range(3):
                lo = np.nextafter(lo, np.float32(0))
                hi = np.nextafter(hi, np.float32(1e30))
                cand += [lo, hi]
        cand = np.array(cand, dtype=np.float32)
        cand[1::2] *= -1                                           # both signs
        for i in range(0, len(cand), 15):
            blk = np.zeros(16, dtype=np.float32)
            blk[0] = np.float32(6.0 * v)                           # the block's largest magnitude
            chunk = cand[i:i + 15]
            blk[1:1 + len(chunk)] = chunk
            blocks.append(blk)
    if len(blocks) % 2:
        blocks.append(np.zeros(16, dtype=np.float32))
    x = np.concatenate(blocks).reshape(-1, 32)
    big = np.zeros((1, 32), dtype=np.float32)
    big[0, 0] = 2688.0                                             # tensor amax: s = 1
    x = np.vstack([big, x])
    _, _, s = Q.quantize_nvfp4(x)
    assert s == np.float32(1.0)
    check("nvfp4", x)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("rows,K,scale_factor", [(200, 96, 1.0), (1000, 512, 1.0), (256, 4096, 0.25),
                                                  (129, 160, 3.0), (128, 256, 0.0)])
def test_nvfp4_given_scale(rows, K, scale_factor, bf16):
    # bsg_quantize_nvfp4_scaled: the recipe's steps 2-3 with the caller's global scale, one pass.
    # Against the oracle's quantize_nvfp4(x, s) bit for bit: the tensor's own s (then also the
    # bytes of bsg_quantize), a quarter of it (many blocks saturate at scale 448 and elements at
    # +-6), three times it (small scales), and 0 (everything zero).
    x = synth.normal_rowscaled(rows, K, seed=rows * 3 + K)
    if bf16:
        bits = synth.as_bf16_bits(x)
        vals = F.decode_bf16(bits).astype(np.float32)
        xd = torch.from_numpy(bits.view(np.int16)).cuda()
    else:
        vals = x
        xd = torch.from_numpy(x).cuda()
    s = np.float32(Q.nvfp4_global_scale(vals) * np.float32(scale_factor))
    sd = torch.tensor([float(s)], dtype=torch.float32, device="cuda")
    codes = torch.full((rows * K // 2,), 0xCD, dtype=torch.uint8, device="cuda")
    sf = torch.full((bsg.bsg_sf_bytes(bsg.BSG_NVFP4, rows, K),), 0xAB, dtype=torch.uint8, device="cuda")
    bsg.bsg_quantize_nvfp4_scaled(xd, rows, K, codes, sf, sd, bf16_input=bf16)
    torch.cuda.synchronize()
    oc, osf, _ = Q.quantize_nvfp4(vals, s)
    assert np.array_equal(codes.cpu().numpy(), oc.ravel())
    assert np.array_equal(sf.cpu().numpy(), L.swizzle(osf))
    assert float(sd.item()) == float(s), "the global scale is read, not written"
    if scale_factor == 1.0:
        c2, sf2, _ = (gpu_quantize_bf16 if bf16 else gpu_quantize)("nvfp4", bits if bf16 else x)
        assert np.array_equal(codes.cpu().numpy(), c2) and np.array_equal(sf.cpu().numpy(), sf2)
    if scale_factor == 0.25:
        sat = ((oc & 0x7) == 0x7) | (((oc >> 4) & 0x7) == 0x7)
        assert (osf == 0x7E).any() and sat.any()   # saturation reached on both levels


def test_nvfp4_given_scale_near_rounding_midpoints():
    # bsg_quantize_nvfp4_scaled against the oracle on the inputs its exact-rational pins use: block
    # amaxes within 3 ulps of every midpoint between neighbouring E4M3 values, and elements within
    # 4 ulps of every E2M1 threshold, for global scales with long significands (both quotients
    # x / den and amax / d land within a rounding of a code boundary).
    e4 = [float(F.E4M3_VALUES[c]) for c in range(0x7F) if np.isfinite(F.E4M3_VALUES[c])]
    mids = [(e4[i] + e4[i + 1]) / 2 for i in range(len(e4) - 1)] + [464.0]
    for s in (np.float32(np.float32(10.3125) / np.float32(2688.0)), np.float32(0.0123456789)):
        d = np.float32(np.float32(6.0) * s)
        rows = []
        for m in mids:                                           # block-scale midpoints
            base = np.float32(np.float64(m) * np.float64(d))
            for k in range(-3, 4):
                v = base
                for _ in range(abs(k)):
                    v = np.nextafter(v, np.float32(np.inf) if k > 0 else np.float32(0))
                blk = np.zeros(16, dtype=np.float32)
                blk[0] = v
                rows.append(blk)
        for code in (0x30, 0x35, 0x3B, 0x41, 0x4E, 0x57):       # element thresholds
            den = np.float32(np.float32(F.E4M3_VALUES[code]) * s)
            cand = []
            for T in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0):
                base = np.float32(np.float32(T) * den)
                for k in range(-4, 5):
                    v = base
                    for _ in range(abs(k)):
                        v = np.nextafter(v, np.float32(np.inf) if k > 0 else np.float32(0))
                    cand.append(v)
            cand = np.array(cand, dtype=np.float32)
            cand[1::2] *= -1
            for i in range(0, len(cand), 15):
                blk = np.zeros(16, dtype=np.float32)
                blk[0] = np.float32(np.float32(6.0) * den)
                chunk = cand[i:i + 15]
                blk[1:1 + len(chunk)] = chunk
                rows.append(blk)
        if len(rows) % 2:
            rows.append(np.zeros(16, dtype=np.float32))
        x = np.stack(rows).reshape(-1, 32)
        nrows, K = x.shape
        sd = torch.tensor([float(s)], dtype=torch.float32, device="cuda")
        codes = torch.full((nrows * K // 2,), 0xCD, dtype=torch.uint8, device="cuda")
        sf = torch.full((bsg.bsg_sf_bytes(bsg.BSG_NVFP4, nrows, K),), 0xAB, dtype=torch.uint8, device="cuda")
        bsg.bsg_quantize_nvfp4_scaled(torch.from_numpy(x).cuda(), nrows, K, codes, sf, sd, bf16_input=False)
        torch.cuda.synchronize()
        oc, osf, _ = Q.quantize_nvfp4(x, s)
        assert np.array_equal(codes.cpu().numpy(), oc.ravel())
        assert np.array_equal(sf.cpu().numpy(), L.swizzle(osf))
