"""Block-scaled FP8 projections (the checkpoint format of section 04 of the Qwen3.8-27B page:
E4M3 weights with one scale per 128 x 128 block, activations quantised per token and 128-wide
group) against the fp64 oracle: the quantisers bit for bit (codes and scales, including every E4M3
rounding boundary), the tcgen05 GEMM element by element over ragged shapes, the K split over
clusters at the layer's decode shapes, the stream-K path at mid-sized token counts, the 128 x 256
wide-tile path at prefill-like token counts, reuse of the workspace without clearing, and
quantise-then-multiply end to end."""
import numpy as np
import pytest
import torch

from oracle import oracle
from tests import gdnutil as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from gated_deltanet_linear_conv1d_gb300 import build
    build.build()
    from gated_deltanet_linear_conv1d_gb300 import binding
    return binding


def _dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).cuda()


@pytest.mark.parametrize("T,K", [(1, 128), (37, 384), (256, 6144), (1000, 5120)])
def test_quant_act_bit_exact(b, T, K):
    rng = np.random.default_rng(200 + T)
    x = rng.normal(size=(T, K)).astype(np.float32) * rng.uniform(0.01, 30.0, size=(T, 1)).astype(np.float32)
    x[0, :128] = 0.0  # an all-zero group
    xb = U.synth.bf16_bits(x)
    x8 = torch.zeros((T, K), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((T, K // 128), dtype=torch.float32, device="cuda")
    b.gdn_fp8_quant_act(U.dev_bf16(xb), x8, xs)
    codes, s = oracle.fp8_quant_act(xb)
    np.testing.assert_array_equal(xs.cpu().numpy(), s)
    np.testing.assert_array_equal(x8.cpu().numpy(), codes)


def _e4m3_boundaries():
    """Every rounding boundary of E4M3 below its largest finite value: midpoints between neighbouring
    codes (subnormal spacing 2^-9 below 2^-6, then 8 steps per binade) with at most 5 significant bits."""
    vals = [(2 * j + 1) * 2.0 ** -10 for j in range(8)]  # 0 .. 2^-6 in steps of 2^-9
    for e in range(-6, 9):
        vals += [(1 + (2 * j + 1) / 16) * 2.0 ** e for j in range(8)]
    return np.array([v for v in vals if v < 448.0])


def test_quant_act_rounding_boundaries(b):
    """x / s landing exactly on E4M3 rounding boundaries (ties to even), once with power-of-two scales
    (x / s exact, and x r exact too) and once with scales 1.25, 1.5, 1.75 times a power of two (x / s
    still exact, x r not: the quotient the kernel multiplies out sits within a rounding of the
    boundary on either side), plus each boundary's bf16 neighbours; codes and scales bit for bit."""
    mids = _e4m3_boundaries()
    rng = np.random.default_rng(77)
    rows = []
    for mult in (1.0, 1.25, 1.5, 1.75):
        for k in (-8, -3, 0, 5):
            sc = mult * 2.0 ** k
            base = (mids * sc).astype(np.float32)
            assert not np.any(base.view(np.uint32) & 0xffff)  # <= 8 significant bits: exact in bf16
            bits = (base.view(np.uint32) >> 16).astype(np.int64)
            for step in (0, 1, -1):  # the boundary, and the bf16 values just above and below it
                g = np.zeros(128, np.uint16)
                g[0] = np.float32(448.0 * sc).view(np.uint32) >> 16  # the group's largest magnitude: s = sc
                body = (bits + step).astype(np.uint16)[:127]
                body |= (rng.integers(0, 2, size=body.size) << 15).astype(np.uint16)  # random signs
                g[1:1 + body.size] = body
                rows.append(g)
    xb = np.array(rows, np.uint16)
    T, K = xb.shape
    x8 = torch.zeros((T, K), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((T, 1), dtype=torch.float32, device="cuda")
    b.gdn_fp8_quant_act(U.dev_bf16(xb), x8, xs)
    codes, s = oracle.fp8_quant_act(xb)
    np.testing.assert_array_equal(xs.cpu().numpy(), s)
    np.testing.assert_array_equal(x8.cpu().numpy(), codes)


@pytest.mark.parametrize("N,K", [(16, 128), (200, 256), (5120, 6144)])
def test_quant_weight_bit_exact(b, N, K):
    rng = np.random.default_rng(300 + N)
    w = (rng.normal(size=(N, K)) / np.sqrt(K)).astype(np.float32)
    wb = U.synth.bf16_bits(w)
    w8 = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(((N + 127) // 128, K // 128), dtype=torch.float32, device="cuda")
    b.gdn_fp8_quant_weight(U.dev_bf16(wb), w8, ws)
    codes, s = oracle.fp8_quant_weight(wb)
    np.testing.assert_array_equal(ws.cpu().numpy(), s)
    np.testing.assert_array_equal(w8.cpu().numpy(), codes)


def _operands(T, K, N, seed):
    """Codes, block scales and a residual of the product's own magnitude (a unit-scale residual
    would dwarf the product, and a wrong product would then still pass)."""
    rng = np.random.default_rng(seed)
    x8 = U.synth.fp8_codes(rng, (T, K))
    w8 = U.synth.fp8_codes(rng, (N, K))
    xs = rng.uniform(0.002, 0.02, size=(T, K // 128)).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-3, size=((N + 127) // 128, K // 128)).astype(np.float32)
    # rms of one product entry: sum over K of two independent codes (rms 2.06 each) times the scales
    prod_rms = np.sqrt(K) * 2.06 * 2.06 * np.sqrt(np.mean(xs ** 2)) * np.sqrt(np.mean(ws ** 2))
    r = U.synth.bf16_bits((rng.normal(size=(T, N)) * prod_rms).astype(np.float32))
    return x8, xs, w8, ws, r


@pytest.mark.parametrize("T,K,N,res,with_ws", [
    (1, 128, 16, False, True),        # one tile, one K block
    (130, 256, 144, True, True),      # ragged m and n tiles
    (300, 1024, 384, False, False),   # no workspace: one K split
    (256, 6144, 5120, True, True),    # Wo at the decode batch: split K
    (256, 5120, 10240, False, True),  # the QKV projection at the decode batch: split K
    (2000, 768, 256, True, True),     # many m tiles
])
def test_fp8_linear_matches_oracle(b, T, K, N, res, with_ws):
    x8, xs, w8, ws, r = _operands(T, K, N, 400 + T + N)
    out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    wsp = torch.zeros(max(256, b.gdn_fp8_linear_workspace_bytes(T, K, N)), dtype=torch.uint8, device="cuda") if with_ws else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.gdn_fp8_linear(_dev_u8(x8), U.dev(xs), _dev_u8(w8), U.dev(ws), out, residual=U.dev_bf16(r) if res else None,
                     workspace=wsp, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    ref = oracle.fp8_linear(x8, xs, w8, ws, r if res else None)
    U.check_out(U.host_f64_from_bf16(out), ref, "out")


def test_fp8_linear_repeat_and_in_place(b):
    """Two calls on one workspace give the same result; out may be the residual itself."""
    T, K, N = 256, 6144, 5120
    x8, xs, w8, ws, r = _operands(T, K, N, 450)
    wsp = torch.zeros(max(256, b.gdn_fp8_linear_workspace_bytes(T, K, N)), dtype=torch.uint8, device="cuda")
    args = (_dev_u8(x8), U.dev(xs), _dev_u8(w8), U.dev(ws))
    out1 = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    out2 = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    b.gdn_fp8_linear(*args, out1, workspace=wsp)
    b.gdn_fp8_linear(*args, out2, workspace=wsp)
    ref = oracle.fp8_linear(x8, xs, w8, ws)
    U.check_out(U.host_f64_from_bf16(out1), ref, "first call")
    U.check_out(U.host_f64_from_bf16(out2), ref, "second call")
    hidden = U.dev_bf16(r)
    b.gdn_fp8_linear(*args, hidden, residual=hidden, workspace=wsp)
    U.check_out(U.host_f64_from_bf16(hidden), oracle.fp8_linear(x8, xs, w8, ws, r), "in place")


def test_quantise_then_multiply_end_to_end(b):
    """bf16 Ogate and Wo quantised on the GPU, multiplied on the GPU, against the oracle doing the
    same steps; and the FP8 result stays within the quantisation error of the bf16 product."""
    T, K, N = 128, 6144, 1024
    rng = np.random.default_rng(460)
    xb = U.synth.bf16_bits(rng.normal(size=(T, K)).astype(np.float32))
    wb = U.synth.bf16_bits((rng.normal(size=(N, K)) / np.sqrt(K)).astype(np.float32))
    x8 = torch.zeros((T, K), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((T, K // 128), dtype=torch.float32, device="cuda")
    w8 = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    ws = torch.zeros((N // 128, K // 128), dtype=torch.float32, device="cuda")
    b.gdn_fp8_quant_act(U.dev_bf16(xb), x8, xs)
    b.gdn_fp8_quant_weight(U.dev_bf16(wb), w8, ws)
    out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    wsp = torch.zeros(max(256, b.gdn_fp8_linear_workspace_bytes(T, K, N)), dtype=torch.uint8, device="cuda")
    b.gdn_fp8_linear(x8, xs, w8, ws, out, workspace=wsp)
    cx, sx = oracle.fp8_quant_act(xb)
    cw, sw = oracle.fp8_quant_weight(wb)
    ref = oracle.fp8_linear(cx, sx, cw, sw)
    U.check_out(U.host_f64_from_bf16(out), ref, "fp8 path")
    exact = oracle.out_proj(xb, wb)
    assert U.rel_l2(ref, exact) < 0.06  # E4M3 keeps 3 mantissa bits: a few percent of quantisation error


@pytest.mark.parametrize("T,K,N,res", [(1, 6144, 5120, True), (16, 256, 144, False), (100, 5120, 6144, True),
                                       (256, 5120, 96 * 2, False), (257, 1024, 256, False)])
def test_fp8_linear_decode_batches(b, T, K, N, res):
    """Decode-sized token counts (one to three m tiles of 128 x 256, each tile's K blocks split over a
    cluster of CTAs that add their parts through the workspace): a single token, ragged tiles, the
    a|b width, and a ragged third m tile; the workspace is reused without clearing."""
    x8, xs, w8, ws, r = _operands(T, K, N, 470 + T + N)
    out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    wsp = torch.zeros(max(256, b.gdn_fp8_linear_workspace_bytes(T, K, N)), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):  # the second call reuses the workspace without clearing it
        b.gdn_fp8_linear(_dev_u8(x8), U.dev(xs), _dev_u8(w8), U.dev(ws), out,
                         residual=U.dev_bf16(r) if res else None, workspace=wsp, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    U.check_out(U.host_f64_from_bf16(out), oracle.fp8_linear(x8, xs, w8, ws, r if res else None), "out")


@pytest.mark.parametrize("T,K,N,res", [
    (4836, 256, 2048, True),    # 38 x 8 = 304 tiles of 128 x 256: the wide tiles, ragged last row tile
    (4836, 384, 2176, False),   # the last column tile's second half lies past N
    (9800, 128, 4096, True),    # one K block, eight tiles per CTA
    (39000, 128, 144, True),    # 305 row tiles of one ragged column tile (N = 144 < 256)
])
def test_fp8_linear_wide_tiles(b, T, K, N, res):
    """Token counts with at least two waves of 128 x 256 tiles take the wide kernel on persistent CTA
    pairs (each pair multiplies 256 tokens x 256 outputs with M = 256 pair MMAs, each CTA folding its
    own 128 rows in registers): ragged rows and columns, a half tile past the last column, an odd
    number of row tiles (the last pair's second CTA has no rows: 9800 and 39000 tokens), several
    tiles per CTA; called twice on the same buffers."""
    x8, xs, w8, ws, r = _operands(T, K, N, 490 + T + N)
    out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    wsp = torch.zeros(max(256, b.gdn_fp8_linear_workspace_bytes(T, K, N)), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        b.gdn_fp8_linear(_dev_u8(x8), U.dev(xs), _dev_u8(w8), U.dev(ws), out,
                         residual=U.dev_bf16(r) if res else None, workspace=wsp, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    U.check_out(U.host_f64_from_bf16(out), oracle.fp8_linear(x8, xs, w8, ws, r if res else None), "out")


@pytest.mark.parametrize("T,K,N,res,with_ws", [
    (129, 2048, 1024, True, True),     # 8 tiles, K split 4 ways; the second m tile holds one live row
    (64, 6144, 5136, False, True),     # 21 tiles, the last one 16 outputs wide; K split 4 ways
    (256, 6144, 5120, True, False),    # Wo at the decode batch without a workspace: one CTA per tile
    (1000, 256, 5120, True, True),     # 160 tiles of 128 x 256: the 128 x 128 kernel, whole tiles
    (12800, 256, 384, False, True),    # 300 tiles of 128 x 128 in two nearly full waves: whole tiles
    (1000, 6144, 5120, True, True),    # Wo, 320 tiles: stream-K, 101 - 102 K blocks (three tiles) per CTA
    (1536, 3072, 5120, False, True),   # 480 tiles: stream-K, ranges holding whole tiles between two pieces
])
def test_fp8_linear_schedules(b, T, K, N, res, with_ws):
    """Each schedule of gdn_fp8_linear on a 152-SM GB300, picked by the number of 128 x 256 output
    tiles: at most one wave splits K over clusters (the parts meet in the workspace, in part order),
    between one and two waves takes 128 x 128 tiles (whole tiles, or stream-K when the last wave of
    whole tiles would leave SMs idle); two calls in a row give the same bits."""
    x8, xs, w8, ws, r = _operands(T, K, N, 520 + T + N)
    wsp = torch.zeros(max(256, b.gdn_fp8_linear_workspace_bytes(T, K, N)), dtype=torch.uint8, device="cuda") if with_ws else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(2):
        out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
        b.gdn_fp8_linear(_dev_u8(x8), U.dev(xs), _dev_u8(w8), U.dev(ws), out,
                         residual=U.dev_bf16(r) if res else None, workspace=wsp, dev_err=err)
        outs.append(out)
    assert b.gdn_read_device_error(err) == 0
    assert torch.equal(outs[0], outs[1])
    U.check_out(U.host_f64_from_bf16(outs[0]), oracle.fp8_linear(x8, xs, w8, ws, r if res else None), "out")


@pytest.mark.parametrize("T", [4836, 4964])
def test_fp8_linear_pairs_in_place(b, T):
    """The CTA-pair schedule with out = residual (the residual stream updated in place): 38 row tiles,
    and 39 (the last pair's second CTA past T); the residual pieces of each stage are loaded before
    its stores, so no store overwrites a residual value still to be read."""
    K, N = 384, 2048
    x8, xs, w8, ws, r = _operands(T, K, N, 530 + T)
    hidden = U.dev_bf16(r)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.gdn_fp8_linear(_dev_u8(x8), U.dev(xs), _dev_u8(w8), U.dev(ws), hidden, residual=hidden, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    U.check_out(U.host_f64_from_bf16(hidden), oracle.fp8_linear(x8, xs, w8, ws, r), "in place")
