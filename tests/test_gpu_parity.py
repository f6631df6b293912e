"""Parity of the CUDA path (through the C ABI) with the CPU oracle, element by element.

Acceptance (per stage):
  * bias_mul_add, token_cat_fp8, token_cat_nvfp4 (codes and block scales), residual_out,
    the V copy of the QKV epilogue: bit-exact.
  * QKV epilogue Q and K: at most one BF16 ulp against the oracle (counts reported).
  * quantise stage: q_gpu == E4M3(RN(y_gpu * inv)) bit-exact for every element (the
    oracle's quantise applied to the GPU's own y).
  * LayerNorm outputs: max |ulp| of y <= 1 against the oracle; q bit-exact wherever y
    matches, at most one E4M3 code step elsewhere.
Every output buffer is canary-guarded (no write outside it).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

MAX_Y_ULP = 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_quant_row_gb300 as fq
    fq.build()
    return fq


def fq():
    import fp8_quant_row_gb300
    return fp8_quant_row_gb300


def check_ln(y_gpu, q_gpu, y_ref, q_ref, input_scale, what=""):
    d = G.bf16_ulp_diff(y_gpu, y_ref)
    nmis = int((d != 0).sum())
    assert d.max(initial=0) <= MAX_Y_ULP, f"{what}: y max ulp {d.max()} ({nmis} mismatches)"
    same = d == 0
    assert np.array_equal(q_gpu[same], q_ref[same]), f"{what}: q differs where y matches"
    assert G.e4m3_step_diff(q_gpu[~same], q_ref[~same]).max(initial=0) <= 1, what
    inv = oracle.recip_f32(input_scale)
    assert np.array_equal(q_gpu, oracle.quantize_array(G.bf16_as_f32(y_gpu), inv)), \
        f"{what}: quantise stage not bit-exact on the GPU's own y"
    from tests.conftest import PARITY_COUNTS
    PARITY_COUNTS.append((what, nmis, int(y_gpu.size)))
    return nmis


def run_nss(inp, input_scale, mod_rows=0, eps=1e-6):
    x = G.dev_bf16(inp["x"])
    rows, cols = inp["x"].shape
    y = G.Guarded((rows, cols), torch.bfloat16)
    q = G.Guarded((rows, cols), torch.float8_e4m3fn)
    fq().nss_fp8(x, G.dev_bf16(inp["scale"]), G.dev_bf16(inp["shift"]), G.dev_scale(input_scale),
                 mod_rows=mod_rows, eps=eps, y=y.tensor, q=q.tensor)
    torch.cuda.synchronize()
    assert y.intact() and q.intact(), "write outside an output buffer"
    assert fq().device_error() == 0, "a bounded wait inside the kernel ran out"
    return G.host_u16(y.tensor), G.host_u8(q.tensor)


# ------------------------------------------------------------------------------------------
# nss_fp8
# ------------------------------------------------------------------------------------------

def test_nss_tiny_config():
    c = W.CONFIGS["nss_tiny"]
    inp = W.config_inputs("nss_tiny")
    yg, qg = run_nss(inp, c["input_scale"])
    yr, qr = oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], c["input_scale"])
    check_ln(yg, qg, yr, qr, c["input_scale"], "nss tiny")


@pytest.mark.parametrize("input_scale", W.QWEN_INPUT_SCALES)
@pytest.mark.parametrize("rows", (1, 127, 1024, 4608))
def test_nss_qwen_sweep(rows, input_scale):
    inp = W.config_inputs("nss_qwen", rows=rows)
    yg, qg = run_nss(inp, input_scale)
    yr, qr = oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], input_scale)
    n = check_ln(yg, qg, yr, qr, input_scale, f"nss qwen rows={rows} s={input_scale}")
    assert n <= max(2, rows // 256)


def test_nss_flux_per_sample_modulation():
    c = W.CONFIGS["nss_flux"]
    inp = W.config_inputs("nss_flux")
    yg, qg = run_nss(inp, c["input_scale"], mod_rows=c["mod_rows"])
    yr, qr = oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], c["input_scale"],
                            mod_rows=c["mod_rows"])
    check_ln(yg, qg, yr, qr, c["input_scale"], "nss flux")


@pytest.mark.parametrize("rows,cols,mod_rows", [
    (1, 8, 0), (3, 16, 0), (5, 24, 2), (7, 1000, 0), (33, 4096, 0), (2, 32768, 0),
    (1, 3072, 0), (2, 3072, 0), (3, 3072, 1), (9, 3072, 4), (1000, 3072, 300),
    (1, 6144, 0), (3, 6144, 0), (17, 6144, 5), (1001, 6144, 500), (300, 6144, 0),
])
def test_nss_shapes_and_ragged_rows(rows, cols, mod_rows):
    n_mod = (rows + mod_rows - 1) // mod_rows if mod_rows else 1
    inp = W.nss_inputs(rows, cols, seed=rows * 7 + cols, n_mod=n_mod, outlier_channels=cols // 100)
    yg, qg = run_nss(inp, 0.05, mod_rows=mod_rows)
    yr, qr = oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], 0.05, mod_rows=mod_rows)
    check_ln(yg, qg, yr, qr, 0.05, f"shape {rows}x{cols}/{mod_rows}")


def test_nss_width_3072_many_rows_per_cta():
    """50 rows per SM: each CTA of the width-3072 kernel refills its row ring more than once
    (a ragged row count and three modulation groups, so CTAs are divided among groups)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = 50 * sms + 37
    mod_rows = (rows + 2) // 3
    inp = W.nss_inputs(rows, 3072, seed=5, n_mod=3, outlier_channels=30)
    yg, qg = run_nss(inp, 0.0625, mod_rows=mod_rows)
    yr, qr = oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], 0.0625, mod_rows=mod_rows)
    check_ln(yg, qg, yr, qr, 0.0625, f"one warp per row, {rows} rows")


def test_nss_more_modulation_groups_than_sms():
    """Every CTA of the tuned kernels serves one modulation group, so a launch with more
    groups than SMs (here one scale/shift row per data row) falls back to the CTA-per-row
    kernel; it must still match the oracle, and so must a launch with exactly one group per
    SM's worth of rows."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for rows, mod_rows in ((2 * sms + 96, 1), (3 * sms, 3), (sms * 10 + 7, 10)):
        n_mod = (rows + mod_rows - 1) // mod_rows
        inp = W.nss_inputs(rows, 3072, seed=rows + mod_rows, n_mod=n_mod, outlier_channels=30)
        yg, qg = run_nss(inp, 0.05, mod_rows=mod_rows)
        yr, qr = oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], 0.05, mod_rows=mod_rows)
        check_ln(yg, qg, yr, qr, 0.05, f"{rows} rows, {n_mod} modulation groups")


def test_nss_kernel_choices_give_identical_bits():
    """The row count picks the kernel (CTA per row up to 2 rows per SM, the warp-specialised
    kernel above) and, inside the latter, how many ring stages a CTA refills (21 stages: the
    refill starts at 22 rows per CTA). Across each boundary the same leading rows must come
    out bit for bit the same."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for n in (2 * sms, 21 * sms, 48 * sms):
        inp = W.nss_inputs(n + 1, 3072, seed=n, outlier_channels=30)
        a = run_nss({k: v[:n] if k == "x" else v for k, v in inp.items()}, 0.0625)
        b = run_nss(inp, 0.0625)
        assert np.array_equal(a[0], b[0][:n]) and np.array_equal(a[1], b[1][:n]), f"{n} vs {n + 1}"


def test_nss_degenerate_rows():
    """Constant rows (var = 0), tiny spreads (var ~ eps), large means, huge values that
    saturate the E4M3 encode, zero rows."""
    cols = 3072
    rng = np.random.default_rng(0)
    rows = []
    bf = lambda v: W.to_bf16_bits(torch.tensor(np.asarray(v, np.float32)))
    rows.append(bf(np.full(cols, 0.75)))
    rows.append(bf(np.zeros(cols)))
    rows.append(bf(rng.standard_normal(cols) * 1e-3))
    rows.append(bf(100.0 + rng.standard_normal(cols) * 0.01))
    rows.append(bf(rng.standard_normal(cols) * 3e4))
    rows.append(bf(np.where(rng.random(cols) < 0.5, -1.0, 1.0)))
    rows.append(bf(rng.standard_normal(cols) * 1e-30))
    x = np.stack(rows)
    g = torch.Generator().manual_seed(1)
    scale = W.normal_bf16((1, cols), 0.1, g)
    shift = W.normal_bf16((1, cols), 0.1, g)
    big_shift = W.normal_bf16((1, cols), 300.0, g)
    for sh in (shift, big_shift):
        for s in (0.0625, 0.0123):
            inp = dict(x=x, scale=scale, shift=sh)
            yg, qg = run_nss(inp, s)
            yr, qr = oracle.nss_fp8(x, scale, sh, s)
            check_ln(yg, qg, yr, qr, s, "degenerate")
    # constant row: n == 0 exactly, so y == shift bitwise
    yg, _ = run_nss(dict(x=x, scale=scale, shift=shift), 0.05)
    assert np.array_equal(yg[0], shift[0]) and np.array_equal(yg[1], shift[0])


def _edge_rows(cols, rng):
    """Rows at the edges of the documented value range (|x| < 2^56, finite): full rows near
    2^55, one element just under 2^56, 2^50 and 2^-50 mixed, bf16 subnormals, values near
    2^-60 (eps dominates), a constant 2^55 row, a large mean with a spread of a few bf16
    steps."""
    bf = lambda v: W.to_bf16_bits(torch.tensor(np.asarray(v, np.float32)))
    z = rng.standard_normal(cols)
    one = z.copy()
    one[cols // 3] = 2.0 ** 55 * 1.9921875  # the largest bf16 below 2^56
    sign = np.where(rng.random(cols) < 0.5, -1.0, 1.0)
    mixed = np.where(rng.random(cols) < 0.5, 2.0 ** 50, 2.0 ** -50) * sign * (1 + rng.random(cols))
    return np.stack([bf(z * 2.0 ** 53), bf(one), bf(mixed), bf(z * 1e-39), bf(z * 2.0 ** -60),
                     bf(np.full(cols, 2.0 ** 55)), bf(2.0 ** 20 + z * 2.0 ** 14)])


@pytest.mark.parametrize("cols", (3072, 6144))
def test_nss_value_range_edges(cols):
    """The edge rows alone (one CTA per row) and tiled among normal rows in a launch large
    enough for the tuned kernels (width 3072: warp-specialised, 6144: two warps per row)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(cols)
    edges = _edge_rows(cols, rng)
    g = torch.Generator().manual_seed(cols)
    scale = W.normal_bf16((1, cols), 0.1, g)
    shift = W.normal_bf16((1, cols), 0.1, g)
    big = W.nss_inputs(2 * sms + 101, cols, seed=cols + 1)["x"]
    big[::37][: len(edges) * 4] = np.tile(edges, (4, 1))[: big[::37].shape[0]]
    for x in (edges, big):
        for s in (0.05, 2.0 ** 50):
            inp = dict(x=x, scale=scale, shift=shift)
            yg, qg = run_nss(inp, s)
            yr, qr = oracle.nss_fp8(x, scale, shift, s)
            check_ln(yg, qg, yr, qr, s, f"value-range edges {x.shape[0]}x{cols} s={s}")


def _mean_on_grid_rows(cols, rng):
    """Rows whose mean lies within 2^-18 |mean| of a bf16 value c while most elements equal c,
    so x - mean is tiny and the per-element |t| < t_small test (exact path) decides: cols - 2
    elements c, one 2c and one c * 2^-20 (mean c (1 + 2^-20 / cols)), for several c and signs;
    also c with five elements a step above and ten half a step below (mean c where the steps
    are bf16 values)."""
    bf = lambda v: W.to_bf16_bits(torch.tensor(np.asarray(v, np.float32)))
    rows = []
    for c in (1.0, -3.0, 0.75 * 2.0 ** 40, -1.5 * 2.0 ** -30, 100.0):
        r = np.full(cols, c)
        idx = rng.permutation(cols)
        r[idx[0]] = 2 * c
        r[idx[1]] = c * 2.0 ** -20
        rows.append(bf(r))
        r = np.full(cols, c)
        step = abs(c) * 2.0 ** -7
        r[idx[:5]] += step
        r[idx[5:15]] -= step / 2
        rows.append(bf(r))
    return np.stack(rows)


@pytest.mark.parametrize("cols", (3072, 6144))
def test_nss_mean_on_a_bf16_value(cols):
    """Rows that take the per-element |t| < t_small exact path, alone and inside a launch large
    enough for the tuned kernels (width 3072: warp-specialised, whose output warps pick the
    code path with that test per row; 6144: two warps per row)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(cols + 7)
    special = _mean_on_grid_rows(cols, rng)
    g = torch.Generator().manual_seed(cols + 7)
    scale = W.normal_bf16((1, cols), 0.1, g)
    shift = W.normal_bf16((1, cols), 0.1, g)
    big = W.nss_inputs(2 * sms + 101, cols, seed=cols + 8)["x"]
    big[5::29][: len(special) * 3] = np.tile(special, (3, 1))[: big[5::29].shape[0]]
    for x in (special, big):
        for s in (0.05, 3.0):
            inp = dict(x=x, scale=scale, shift=shift)
            yg, qg = run_nss(inp, s)
            yr, qr = oracle.nss_fp8(x, scale, shift, s)
            check_ln(yg, qg, yr, qr, s, f"mean on a bf16 value {x.shape[0]}x{cols} s={s}")


def test_nss_row_pieces_reproduce_the_single_call():
    """A FLUX.2-shaped launch (two modulation groups) cut for 3 and 8 ranks into pieces that
    lie inside one group (each a call with mod_rows = 0 and its group's scale/shift rows):
    the pieces together give the single call's outputs."""
    c = W.CONFIGS["nss_flux"]
    inp = W.config_inputs("nss_flux")
    yr, qr = oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], c["input_scale"],
                            mod_rows=c["mod_rows"])
    for world in (3, 8):
        yp = np.empty_like(yr)
        qp = np.empty_like(qr)
        for rank in range(world):
            for r0, r1, grp in fq().row_pieces(inp["x"].shape[0], c["mod_rows"], world, rank):
                piece = dict(x=inp["x"][r0:r1], scale=inp["scale"][grp:grp + 1],
                             shift=inp["shift"][grp:grp + 1])
                yp[r0:r1], qp[r0:r1] = run_nss(piece, c["input_scale"])
        check_ln(yp, qp, yr, qr, c["input_scale"], f"row pieces for {world} ranks")


def test_pdl_producer_consumer_chains_on_one_stream():
    """Every launch allows programmatic dependent launch and every kernel waits for the
    grids it depends on before its first global access. Chains on one stream with no
    synchronisation in between, each consumer reading what the kernel just before it wrote
    (the destinations hold stale values first, so reading too early shows):
    bias_mul_add -> nss_fp8; scale_residual_nss_fp8 in place -> nss_fp8 on the updated
    residual; nss_fp8 -> nss_fp8 on its y; a torch elementwise kernel -> nss_fp8; a torch
    elementwise kernel -> token_cat_fp8."""
    c = W.CONFIGS["scale_residual_qwen"]
    r = W.config_inputs("scale_residual_qwen")
    s = c["input_scale"]
    x, res = G.dev_bf16(r["x"]), G.dev_bf16(r["residual"])
    bias, gate = G.dev_bf16(r["bias"]), G.dev_bf16(r["gate"])
    scale, shift = G.dev_bf16(r["scale"]), G.dev_bf16(r["shift"])
    ds = G.dev_scale(s)
    x1_ref = oracle.bias_mul_add(r["x"], r["bias"], r["gate"][0], r["residual"])
    y1_ref, q1_ref = oracle.nss_fp8(x1_ref, r["scale"], r["shift"], s)
    ro_ref, _, _ = oracle.scale_residual_nss_fp8(r["x"], r["residual"], r["bias"], r["gate"],
                                                 r["scale"], r["shift"], s)
    y2_ref, q2_ref = oracle.nss_fp8(ro_ref, r["scale"], r["shift"], s)
    y3_ref, q3_ref = oracle.nss_fp8(y1_ref, r["scale"], r["shift"], s)
    t = W.config_inputs("token_cat_flux")
    tc = W.CONFIGS["token_cat_flux"]
    qc_ref = oracle.token_cat_fp8(t["a"], t["m"], tc["input_scale"])
    a_src, m = G.dev_bf16(t["a"]), G.dev_bf16(t["m"])
    a = torch.zeros_like(a_src)
    x_copy = torch.zeros_like(x)
    for rep in range(3):
        x1 = torch.zeros_like(x)
        resid = res.clone()
        torch.cuda.synchronize()
        fq().bias_mul_add(x, bias, gate[0], res, y=x1)
        y1, q1 = fq().nss_fp8(x1, scale, shift, ds)
        fq().scale_residual_nss_fp8(x, resid, gate, scale, shift, ds, bias=bias,
                                    residual_out=resid)
        y2, q2 = fq().nss_fp8(resid, scale, shift, ds)
        y3, q3 = fq().nss_fp8(y1, scale, shift, ds)
        x_copy.zero_()
        torch.mul(x1, 1, out=x_copy)  # an elementwise torch kernel as the producer
        y4, q4 = fq().nss_fp8(x_copy, scale, shift, ds)
        a.zero_()
        torch.mul(a_src, 1, out=a)
        qc = fq().token_cat_fp8(a, m, G.dev_scale(tc["input_scale"]))
        torch.cuda.synchronize()
        assert fq().device_error() == 0, f"rep {rep}: a bounded wait inside a kernel ran out"
        assert np.array_equal(G.host_u16(x1), x1_ref), f"rep {rep}: bias_mul_add"
        assert np.array_equal(G.host_u16(resid), ro_ref), f"rep {rep}: in-place residual"
        for yg, qg, yr_, qr_, what in ((y1, q1, y1_ref, q1_ref, "after bias_mul_add"),
                                       (y2, q2, y2_ref, q2_ref, "after in-place residual"),
                                       (y3, q3, y3_ref, q3_ref, "on the previous y"),
                                       (y4, q4, y1_ref, q1_ref, "after a torch copy")):
            check_ln(G.host_u16(yg), G.host_u8(qg), yr_, qr_, s, f"PDL chain {what} rep {rep}")
        assert np.array_equal(G.host_u8(qc), qc_ref), f"rep {rep}: token_cat after a torch copy"


def test_pdl_chains_qkv_and_nvfp4_on_one_stream():
    """As above for the warp-specialised QKV epilogue and token_cat_nvfp4, on one stream with
    no synchronisation in between: a torch elementwise kernel writes the packed QKV rows ->
    qkv_epilogue -> a second qkv_epilogue whose q, k, v are the first one's outputs; a torch
    elementwise kernel writes the attention part -> token_cat_nvfp4. The oracle's composition
    is the reference."""
    H, tt, it = 24, 64, 300
    d = W.qkv_inputs(tt, it, H, seed=7)
    T = tt + it
    r1 = oracle.qkv_epilogue(d["txt"], d["img"], H)

    def second(lo, hi, st, arrs):
        return dict(q=arrs[0][lo:hi].reshape(hi - lo, H * 128),
                    k=arrs[1][lo:hi].reshape(hi - lo, H * 128),
                    v=arrs[2][lo:hi].reshape(hi - lo, H * 128),
                    wq=st["wq"], wk=st["wk"], cos_sin=st["cos_sin"], eps=st["eps"])

    r2 = oracle.qkv_epilogue(second(0, tt, d["txt"], r1), second(tt, T, d["img"], r1), H)
    srcs = {k: G.dev_bf16(d[k]["packed"]) for k in ("txt", "img")}
    c = W.CONFIGS["token_cat_nvfp4_flux"]
    t = W.config_inputs("token_cat_nvfp4_flux")
    rows = 512
    qn_ref, sn_ref = oracle.token_cat_nvfp4(t["a"][:rows], t["m"][:rows], c["global_scale"])
    a_src, m = G.dev_bf16(t["a"][:rows]), G.dev_bf16(t["m"][:rows])
    a = torch.zeros_like(a_src)
    gs = G.dev_scale(c["global_scale"])
    for rep in range(3):
        packed = {k: torch.zeros_like(v) for k, v in srcs.items()}
        torch.cuda.synchronize()
        for k in packed:
            torch.mul(srcs[k], 1, out=packed[k])  # an elementwise torch kernel as the producer
        o1 = fq().qkv_epilogue(_dev_stream(d["txt"], H, packed["txt"]),
                               _dev_stream(d["img"], H, packed["img"]), H)

        def dev_second(lo, hi, st):
            return dict(q=o1[0][lo:hi].view(hi - lo, H * 128), k=o1[1][lo:hi].view(hi - lo, H * 128),
                        v=o1[2][lo:hi].view(hi - lo, H * 128), q_weight=G.dev_bf16(st["wq"]),
                        k_weight=G.dev_bf16(st["wk"]),
                        cos_sin=torch.from_numpy(st["cos_sin"]).cuda(), eps=st["eps"])

        txt2, img2 = dev_second(0, tt, d["txt"]), dev_second(tt, T, d["img"])
        o2 = fq().qkv_epilogue(txt2, img2, H)
        a.zero_()
        torch.mul(a_src, 1, out=a)
        qn, sn = fq().token_cat_nvfp4(a, m, gs)
        torch.cuda.synchronize()
        assert fq().device_error() == 0, f"rep {rep}: a bounded wait inside a kernel ran out"
        for name, got, ref in zip("qkv", o1, r1):
            assert np.array_equal(G.host_u16(got), ref), f"rep {rep}: first qkv {name}"
        for name, got, ref in zip("qkv", o2, r2):
            assert np.array_equal(G.host_u16(got), ref), f"rep {rep}: chained qkv {name}"
        assert np.array_equal(G.host_u8(qn), qn_ref), f"rep {rep}: token_cat_nvfp4 codes"
        assert np.array_equal(G.host_u8(sn), sn_ref), f"rep {rep}: token_cat_nvfp4 scales"


def test_nss_eps_values():
    inp = W.nss_inputs(64, 3072, seed=3)
    for eps in (0.0, 1e-6, 1e-2):
        yg, qg = run_nss(inp, 0.05, eps=eps)
        yr, qr = oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], 0.05, eps=eps)
        check_ln(yg, qg, yr, qr, 0.05, f"eps={eps}")


# ------------------------------------------------------------------------------------------
# scale_residual_nss_fp8 and bias_mul_add
# ------------------------------------------------------------------------------------------

def run_scale_residual(inp, input_scale, with_bias=True, in_place=False, mod_rows=0):
    rows, cols = inp["x"].shape
    x = G.dev_bf16(inp["x"])
    res = G.dev_bf16(inp["residual"])
    y = G.Guarded((rows, cols), torch.bfloat16)
    q = G.Guarded((rows, cols), torch.float8_e4m3fn)
    ro = None if in_place else G.Guarded((rows, cols), torch.bfloat16)
    bias = G.dev_bf16(inp["bias"]) if with_bias else None
    r_out, _, _ = fq().scale_residual_nss_fp8(
        x, res, G.dev_bf16(inp["gate"]), G.dev_bf16(inp["scale"]), G.dev_bf16(inp["shift"]),
        G.dev_scale(input_scale), bias=bias, mod_rows=mod_rows,
        residual_out=res if in_place else ro.tensor, y=y.tensor, q=q.tensor)
    torch.cuda.synchronize()
    assert y.intact() and q.intact() and (in_place or ro.intact())
    return G.host_u16(r_out), G.host_u16(y.tensor), G.host_u8(q.tensor)


@pytest.mark.parametrize("with_bias", (True, False))
def test_scale_residual_qwen_config(with_bias):
    c = W.CONFIGS["scale_residual_qwen"]
    inp = W.config_inputs("scale_residual_qwen")
    rg, yg, qg = run_scale_residual(inp, c["input_scale"], with_bias=with_bias)
    rr, yr, qr = oracle.scale_residual_nss_fp8(inp["x"], inp["residual"],
                                               inp["bias"] if with_bias else None, inp["gate"],
                                               inp["scale"], inp["shift"], c["input_scale"])
    assert np.array_equal(rg, rr), "residual_out must be bit-exact"
    check_ln(yg, qg, yr, qr, c["input_scale"], f"scale-residual bias={with_bias}")


def test_scale_residual_in_place_and_shapes():
    for rows, cols, mod_rows in ((37, 3072, 0), (20, 6144, 7), (5, 1024, 0), (3, 40, 1)):
        n_mod = (rows + mod_rows - 1) // mod_rows if mod_rows else 1
        inp = W.residual_inputs(rows, cols, seed=rows + cols, n_mod=n_mod)
        rg, yg, qg = run_scale_residual(inp, 0.05, in_place=True, mod_rows=mod_rows)
        rr, yr, qr = oracle.scale_residual_nss_fp8(inp["x"], inp["residual"], inp["bias"],
                                                   inp["gate"], inp["scale"], inp["shift"], 0.05,
                                                   mod_rows=mod_rows)
        assert np.array_equal(rg, rr)
        check_ln(yg, qg, yr, qr, 0.05, f"in-place {rows}x{cols}")


def test_bias_mul_add_qwen_config_bit_exact():
    inp = W.config_inputs("bias_mul_add_qwen")
    rows, cols = inp["x"].shape
    y = G.Guarded((rows, cols), torch.bfloat16)
    fq().bias_mul_add(G.dev_bf16(inp["x"]), G.dev_bf16(inp["bias"]), G.dev_bf16(inp["gate"][0]),
                      G.dev_bf16(inp["residual"]), y=y.tensor)
    torch.cuda.synchronize()
    assert y.intact()
    ref = oracle.bias_mul_add(inp["x"], inp["bias"], inp["gate"][0], inp["residual"])
    assert np.array_equal(G.host_u16(y.tensor), ref)


def test_bias_mul_add_tie_cases_and_page_example():
    """The page's extreme-value row, exact product ties with +/-/0 residuals, wide exponent
    gaps, and in-place outputs."""
    import json, os
    ex = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "bias_fma_tie_example.json")))["inputs"]
    cols = 64
    rng = np.random.default_rng(5)
    bf = lambda v: W.to_bf16_bits(torch.tensor(np.asarray(v, np.float32)))
    x = bf(rng.standard_normal((4, cols)) * 2.0 ** rng.integers(-20, 20, (4, cols)))
    r = bf(rng.standard_normal((4, cols)) * 2.0 ** rng.integers(-20, 20, (4, cols)))
    b = bf(rng.standard_normal(cols) * 2.0 ** rng.integers(-20, 20, cols))
    g = bf(rng.standard_normal(cols) * 2.0 ** rng.integers(-20, 20, cols))
    x[0, 0], b[0], g[0], r[0, 0] = bf([ex["x"], ex["bias"], ex["gate"], ex["residual"]])
    # exact ties: significand pairs whose product sits on a bf16 midpoint; the residual is
    # zero or a tiny +- value that must break the tie
    from tests.exact import bf16_product_ties
    ties = bf16_product_ties()
    for j in range(1, cols):
        m1, m2 = ties[(j * 37) % len(ties)]
        x[1, j] = bf((-1) ** j * m1 * 2.0 ** (j % 7 - 7))
        b[j] = bf(0.0)
        g[j] = bf(m2 * 2.0 ** -(j % 5 + 7))
        r[1, j] = bf([0.0, 2.0 ** -30, -(2.0 ** -30)][j % 3])
    ref = oracle.bias_mul_add(x, b, g, r)
    for mode in ("fresh", "into_x", "into_residual"):
        xd, rd = G.dev_bf16(x), G.dev_bf16(r)
        out = {"fresh": None, "into_x": xd, "into_residual": rd}[mode]
        y = fq().bias_mul_add(xd, G.dev_bf16(b), G.dev_bf16(g), rd, y=out)
        torch.cuda.synchronize()
        assert np.array_equal(G.host_u16(y), ref), mode
    assert G.bf16_as_f32(ref[0:1, 0:1])[0, 0] == -5079040.0


# ------------------------------------------------------------------------------------------
# token_cat_fp8
# ------------------------------------------------------------------------------------------

def run_token_cat(a, m, s):
    rows = a.shape[0]
    q = G.Guarded((rows, a.shape[1] + m.shape[1]), torch.float8_e4m3fn)
    fq().token_cat_fp8(G.dev_bf16(a), G.dev_bf16(m), G.dev_scale(s), q=q.tensor)
    torch.cuda.synchronize()
    assert q.intact()
    return G.host_u8(q.tensor)


def test_token_cat_flux_config_bit_exact():
    c = W.CONFIGS["token_cat_flux"]
    inp = W.config_inputs("token_cat_flux")
    qg = run_token_cat(inp["a"], inp["m"], c["input_scale"])
    qr = oracle.token_cat_fp8(inp["a"], inp["m"], c["input_scale"])
    assert np.array_equal(qg, qr)


@pytest.mark.parametrize("rows,a_cols,m_cols", [(1, 6144, 18432), (127, 6144, 18432),
                                                (3, 16, 16), (5, 48, 80), (9, 1024, 16)])
def test_token_cat_shapes(rows, a_cols, m_cols):
    inp = W.token_cat_inputs(rows, a_cols, m_cols, seed=rows)
    for s in (0.1, 0.0625, 0.4754464328):
        assert np.array_equal(run_token_cat(inp["a"], inp["m"], s),
                              oracle.token_cat_fp8(inp["a"], inp["m"], s))


def test_token_cat_special_values():
    """+-Inf saturate, NaN encodes 0x7F, -0 and bf16 subnormals, exact E4M3 midpoints."""
    specials = np.array([0x7F80, 0xFF80, 0x7FC0, 0x8000, 0x0000, 0x0001, 0x8001, 0x007F,
                         0x7F7F, 0xFF7F, 0x3F80, 0xBF80], np.uint16)
    mids = []
    for c in range(0x7E):
        v = np.float32((oracle.e4m3_decode(c) + oracle.e4m3_decode(c + 1)) / 2)
        mids.append(int(W.to_bf16_bits(torch.tensor([v]))[0]))
    vals = np.concatenate([specials, np.array(mids, np.uint16), np.array(mids, np.uint16) | 0x8000])
    vals = np.resize(vals, 2 * 256).reshape(2, 256)
    q = run_token_cat(vals[:, :128].copy(), vals[:, 128:].copy(), 1.0)
    ref = oracle.token_cat_fp8(vals[:, :128], vals[:, 128:], 1.0)
    assert np.array_equal(q, ref)


# ------------------------------------------------------------------------------------------
# token_cat_nvfp4
# ------------------------------------------------------------------------------------------

def run_token_cat_nvfp4(a, m, g):
    rows = a.shape[0]
    cols = a.shape[1] + m.shape[1]
    q = G.Guarded((rows, cols // 2), torch.uint8)
    sf = G.Guarded((fq().nvfp4_scale_bytes(rows, cols),), torch.uint8)  # canary-filled too
    fq().token_cat_nvfp4(G.dev_bf16(a), G.dev_bf16(m), G.dev_scale(g), q=q.tensor, sf=sf.tensor)
    torch.cuda.synchronize()
    assert q.intact() and sf.intact()
    return G.host_u8(q.tensor), G.host_u8(sf.tensor)


def check_nvfp4(a, m, g, what=""):
    qg, sg = run_token_cat_nvfp4(a, m, g)
    qr, sr = oracle.token_cat_nvfp4(a, m, g)
    assert np.array_equal(sg, sr), f"{what}: block scales differ at {np.nonzero(sg != sr)[0][:8]}"
    bad = np.nonzero(qg != qr)
    assert not bad[0].size, f"{what}: codes differ at {list(zip(*bad))[:8]}"


def test_token_cat_nvfp4_flux_config_bit_exact():
    c = W.CONFIGS["token_cat_nvfp4_flux"]
    inp = W.config_inputs("token_cat_nvfp4_flux")
    check_nvfp4(inp["a"], inp["m"], c["global_scale"], "flux config")


@pytest.mark.parametrize("rows,a_cols,m_cols", [(1, 6144, 18432), (17, 6144, 18432),
                                                (129, 6144, 18432), (127, 64, 64),
                                                (5, 64, 1024), (300, 128, 192),
                                                # the register-capped one-wave build
                                                (512, 6144, 18432), (333, 6144, 18432)])
def test_token_cat_nvfp4_shapes_and_padding(rows, a_cols, m_cols):
    inp = W.token_cat_inputs(rows, a_cols, m_cols, seed=rows + 7)
    for g in (60.0, 1.0, 358.4, 1e-3, 1e6):
        check_nvfp4(inp["a"], inp["m"], g, f"{rows}x{a_cols}+{m_cols} g={g}")


def test_token_cat_nvfp4_more_row_groups_than_one_grid_dimension():
    """600,000 rows = 75,000 eight-row groups: more than the 65,535 a grid dimension holds, so
    the kernel's row-group loop strides (the pages' wrapper stops at 65,408 rows)."""
    rows = 600_000
    inp = W.token_cat_inputs(rows, 64, 64, seed=9)
    check_nvfp4(inp["a"], inp["m"], 60.0, "600k rows")


def test_token_cat_nvfp4_special_values_and_ties():
    """Exact E2M1 midpoints (ties to even), signed zeros, +-Inf, bf16 subnormals and the
    largest finite bf16, block scales that saturate or vanish."""
    def bf(v):
        return int(W.to_bf16_bits(torch.tensor([float(v)]))[0])
    grid = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    mids = [(x + y) / 2 for x, y in zip(grid, grid[1:])]
    groups = []
    for e in (-4, 0, 3):  # amax 6 * 2^e with g = 1 makes the block scale exactly 2^e
        for sign in (1, -1):
            vals = [6.0] + [sign * v for v in mids] + [sign * v for v in grid[1:]] + [-0.0]
            groups.append([bf(v * 2.0 ** e) for v in vals])
    groups.append([0x7F80, 0xFF80] + [bf(1.0)] * 14)            # +-Inf: scale saturates
    groups.append([0x7F7F, 0xFF7F] + [0x0001] * 14)             # largest finite, subnormals
    groups.append([0x8001, 0x0001, 0x8000, 0x0000] * 4)         # scale code 0: signed zeros
    groups.append([bf(-1e-3)] * 8 + [bf(1e-3)] * 8)
    groups.append([0x8000] * 16)
    groups.append([bf(v) for v in np.linspace(-3, 3, 16)])
    flat = np.array(groups, np.uint16).ravel()
    flat = np.resize(flat, 4 * 128)  # four rows of 128 = 64 + 64
    x = flat.reshape(4, 128)
    for g in (1.0, 0.5, 3.0e4):
        check_nvfp4(x[:, :64].copy(), x[:, 64:].copy(), g, f"specials g={g}")


def test_token_cat_nvfp4_zero_rows_and_repeat_calls_agree():
    inp = W.token_cat_inputs(256, 6144, 18432, seed=3)
    a = inp["a"].copy()
    a[5] = 0
    a[200] = 0x8000
    q1, s1 = run_token_cat_nvfp4(a, inp["m"], 60.0)
    q2, s2 = run_token_cat_nvfp4(a, inp["m"], 60.0)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
    qr, sr = oracle.token_cat_nvfp4(a, inp["m"], 60.0)
    assert np.array_equal(q1, qr) and np.array_equal(s1, sr)


# ------------------------------------------------------------------------------------------
# QKV epilogue
# ------------------------------------------------------------------------------------------

def _dev_stream(st, heads, packed_dev=None):
    """Device tensors for one stream: q, k, v as column slices of one packed tensor."""
    packed = G.dev_bf16(st["packed"]) if packed_dev is None else packed_dev
    hd = heads * 128
    return dict(q=packed[:, :hd], k=packed[:, hd:2 * hd], v=packed[:, 2 * hd:3 * hd],
                q_weight=G.dev_bf16(st["wq"]), k_weight=G.dev_bf16(st["wk"]),
                cos_sin=torch.from_numpy(st["cos_sin"]).cuda(), eps=st["eps"])


def run_qkv(d, heads):
    tt, it = d["txt"]["q"].shape[0], d["img"]["q"].shape[0]
    outs = [G.Guarded((tt + it, heads, 128), torch.bfloat16) for _ in range(3)]
    fq().qkv_epilogue(_dev_stream(d["txt"], heads), _dev_stream(d["img"], heads), heads,
                      out=tuple(o.tensor for o in outs))
    torch.cuda.synchronize()
    assert all(o.intact() for o in outs)
    return [G.host_u16(o.tensor) for o in outs]


def check_qkv(d, heads, what=""):
    gq, gk, gv = run_qkv(d, heads)
    rq, rk, rv = oracle.qkv_epilogue(d["txt"], d["img"], heads)
    assert np.array_equal(gv, rv), f"{what}: v copy differs"
    from tests.conftest import PARITY_COUNTS
    for name, g_, r_ in (("q", gq, rq), ("k", gk, rk)):
        diff = G.bf16_ulp_diff(g_, r_)
        nmis = int((diff != 0).sum())
        assert diff.max(initial=0) <= MAX_Y_ULP, f"{what} {name}: max ulp {diff.max()} ({nmis})"
        PARITY_COUNTS.append((f"qkv {what} {name}", nmis, int(g_.size)))


@pytest.mark.parametrize("name", ["qkv_qwen", "qkv_flux"])
def test_qkv_epilogue_configs(name):
    c = W.CONFIGS[name]
    check_qkv(W.config_inputs(name), c["heads"], name)


@pytest.mark.parametrize("tt,it,heads,extra", [(0, 64, 24, 0), (37, 0, 24, 0), (3, 5, 1, 16),
                                               (2, 9, 5, 48), (7, 4, 7, 0), (1, 1, 13, 16),
                                               (16, 16, 96, 0), (5, 11, 64, 16), (4, 7, 57, 0),
                                               (3, 6, 65, 0)])
def test_qkv_epilogue_shapes(tt, it, heads, extra):
    d = W.qkv_inputs(tt, it, heads, seed=tt * 31 + it + heads, extra_cols=extra)
    d["img"]["eps"] = 1e-5
    check_qkv(d, heads, f"{tt}+{it}x{heads}")


@pytest.mark.parametrize("tt,it,heads", [(300, 1700, 64), (100, 6000, 1), (50, 2000, 33)])
def test_qkv_epilogue_stage_reuse(tt, it, heads):
    """Enough tokens per CTA that every stage of the warp-specialised kernel's ring is reused
    several times: 64 heads (4 stages of 48.5 KB, 13 tokens per CTA), 1 head (32 stages,
    ~40 tokens per CTA), 33 heads (the 13-warp variant, a partial block of eight heads)."""
    check_qkv(W.qkv_inputs(tt, it, heads, seed=heads + 101), heads, f"reuse {tt}+{it}x{heads}")


def test_qkv_epilogue_special_heads():
    """Zero heads, constant heads, tiny and huge magnitudes, exact midpoint products,
    right-angle and identity rotations."""
    heads = 8
    d = W.qkv_inputs(3, 6, heads, seed=77)
    for st in (d["txt"], d["img"]):
        p = st["packed"]
        q = p[:, :heads * 128].reshape(p.shape[0], heads, 128)
        q[0, 0] = 0                                    # all-zero head (eps only)
        q[0, 1] = W.to_bf16_bits(torch.tensor([1.5]))[0]   # constant head
        q[1, 2] = W.to_bf16_bits(torch.randn(128) * 1e-12)
        q[1, 3] = W.to_bf16_bits(torch.randn(128) * 1e15)
        q[2, 4] = 0x8000                               # all -0
        st["q"], st["k"], st["v"] = (p[:, :heads * 128], p[:, heads * 128:2 * heads * 128],
                                     p[:, 2 * heads * 128:3 * heads * 128])
        cs = st["cos_sin"]
        cs[0, :64], cs[0, 64:] = 1.0, 0.0              # identity
        cs[1, :64], cs[1, 64:] = 0.0, 1.0              # 90 degrees
    check_qkv(d, heads, "specials")


def test_qkv_epilogue_repeat_calls_agree():
    d = W.config_inputs("qkv_qwen")
    a = run_qkv(d, 24)
    b = run_qkv(d, 24)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


# ------------------------------------------------------------------------------------------
# boundary behaviour on the device
# ------------------------------------------------------------------------------------------

def test_rows_zero_launches_nothing_and_returns_ok():
    L = fq()._capi.lib()
    assert L.fp8q_nss_fp8(None, None, None, None, None, 0, None, 0, 3072, 1e-6, None) == 0
    assert L.fp8q_token_cat_fp8(None, None, 16, None, 16, None, 0, None) == 0
    assert L.fp8q_token_cat_nvfp4(None, None, None, 64, None, 64, None, 0, None) == 0


def test_errors_are_reported_before_launch():
    L = fq()._capi.lib()
    x = torch.zeros(4, 3072, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    q = torch.empty(4, 3072, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(3072, dtype=torch.bfloat16, device="cuda")
    s = G.dev_scale(1.0)
    args = lambda **kw: [kw.get("y", y.data_ptr()), kw.get("q", q.data_ptr()),
                         kw.get("x", x.data_ptr()), sc.data_ptr(), sc.data_ptr(), 0, s.data_ptr(),
                         kw.get("rows", 4), kw.get("cols", 3072), kw.get("eps", 1e-6), None]
    assert L.fp8q_nss_fp8(*args()) == 0
    assert L.fp8q_nss_fp8(*args(x=x.data_ptr() + 2)) == 2
    assert L.fp8q_nss_fp8(*args(y=x.data_ptr())) == 5
    assert L.fp8q_nss_fp8(*args(cols=3070)) == 3
    assert L.fp8q_nss_fp8(*args(eps=-1.0)) == 7
    torch.cuda.synchronize()


def test_runs_on_a_side_stream_and_is_deterministic():
    inp = W.config_inputs("nss_qwen", rows=512)
    x, sc, sh, s = (G.dev_bf16(inp["x"]), G.dev_bf16(inp["scale"]), G.dev_bf16(inp["shift"]),
                    G.dev_scale(0.25))
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        y1, q1 = fq().nss_fp8(x, sc, sh, s)
    st.synchronize()
    y2, q2 = fq().nss_fp8(x, sc, sh, s)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(q1.view(torch.uint8), q2.view(torch.uint8))


def test_calls_capture_into_a_cuda_graph_and_replay():
    """Every entry point is asynchronous on the given stream and allocates nothing, so it can
    be captured into a CUDA graph; replays on new inputs (copied into the captured buffers)
    must equal direct calls."""
    lib = fq()
    rng_inputs = [W.config_inputs("nss_qwen", rows=256, seed=s) for s in (11, 12)]
    x = G.dev_bf16(rng_inputs[0]["x"])
    sc, sh = G.dev_bf16(rng_inputs[0]["scale"]), G.dev_bf16(rng_inputs[0]["shift"])
    s = G.dev_scale(0.25)
    y = torch.empty_like(x)
    q = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device="cuda")
    t = W.token_cat_inputs(128, 6144, 18432, seed=5)
    a, m = G.dev_bf16(t["a"]), G.dev_bf16(t["m"])
    g = G.dev_scale(60.0)
    q4 = torch.empty(128, 12288, dtype=torch.uint8, device="cuda")
    sf = torch.empty(lib.nvfp4_scale_bytes(128, 24576), dtype=torch.uint8, device="cuda")
    d = W.qkv_inputs(8, 32, 24, seed=6)
    txt, img = _dev_stream(d["txt"], 24), _dev_stream(d["img"], 24)
    jo = tuple(torch.empty(40, 24, 128, dtype=torch.bfloat16, device="cuda") for _ in range(3))

    def calls():
        lib.nss_fp8(x, sc, sh, s, y=y, q=q)
        lib.token_cat_nvfp4(a, m, g, q=q4, sf=sf)
        lib.qkv_epilogue(txt, img, 24, out=jo)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls()  # warm-up outside capture (occupancy queries, attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls()
    # new inputs into the captured buffers, replay, compare with direct calls
    x.copy_(G.dev_bf16(rng_inputs[1]["x"]))
    a.copy_(G.dev_bf16(W.token_cat_inputs(128, 6144, 18432, seed=7)["a"]))
    graph.replay()
    torch.cuda.synchronize()
    got = [G.host_u16(y), G.host_u8(q), G.host_u8(q4), G.host_u8(sf)] + [G.host_u16(o) for o in jo]
    y2, q2 = lib.nss_fp8(x, sc, sh, s)
    q42, sf2 = lib.token_cat_nvfp4(a, m, g)
    jo2 = lib.qkv_epilogue(txt, img, 24)
    torch.cuda.synchronize()
    want = [G.host_u16(y2), G.host_u8(q2), G.host_u8(q42), G.host_u8(sf2)] + [G.host_u16(o) for o in jo2]
    for i, (u, v) in enumerate(zip(got, want)):
        assert np.array_equal(u, v), i
    assert not np.array_equal(got[0], G.host_u16(G.dev_bf16(rng_inputs[0]["x"])))  # really replayed


# ------------------------------------------------------------------------------------------
# seeded random sweeps: shapes, row counts across the kernel choices, scales, eps, value
# ranges and modulation groups drawn from a fixed seed (the same cases on every run)
# ------------------------------------------------------------------------------------------

def _random_scale(rng):
    return float(np.float32(10 ** rng.uniform(-2.5, 0.5)))


def test_random_sweep_nss():
    rng = np.random.default_rng(2026)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for case in range(24):
        cols = int(rng.choice([3072, 6144, 8 * int(rng.integers(1, 600))]))
        tuned = cols in (3072, 6144)
        rows = int(rng.integers(1, 6 * sms if tuned else 300))  # across the 2-rows-per-SM split
        mod_rows = 0 if rng.random() < 0.5 else max(1, rows // int(rng.integers(1, 4)))
        n_mod = (rows + mod_rows - 1) // mod_rows if mod_rows else 1
        s, eps = _random_scale(rng), float(rng.choice([1e-6, 1e-5, 0.0]))
        inp = W.nss_inputs(rows, cols, seed=1000 + case, n_mod=n_mod,
                           outlier_channels=int(rng.integers(0, cols // 50 + 1)),
                           x_std=float(10 ** rng.uniform(-3, 2)))
        yg, qg = run_nss(inp, s, mod_rows=mod_rows, eps=eps)
        yr, qr = oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], s, mod_rows=mod_rows,
                                eps=eps)
        check_ln(yg, qg, yr, qr, s, f"random {case}: {rows}x{cols}/{mod_rows} s={s} eps={eps}")


def test_random_sweep_scale_residual_and_bias_mul_add():
    rng = np.random.default_rng(2027)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for case in range(12):
        cols = int(rng.choice([3072, 6144, 8 * int(rng.integers(1, 400))]))
        rows = int(rng.integers(1, 6 * sms if cols in (3072, 6144) else 200))
        mod_rows = 0 if rng.random() < 0.5 else max(1, rows // int(rng.integers(1, 4)))
        n_mod = (rows + mod_rows - 1) // mod_rows if mod_rows else 1
        with_bias, in_place, s = bool(rng.random() < 0.7), bool(rng.random() < 0.3), _random_scale(rng)
        inp = W.residual_inputs(rows, cols, seed=2000 + case, n_mod=n_mod)
        rg, yg, qg = run_scale_residual(inp, s, with_bias=with_bias, in_place=in_place,
                                        mod_rows=mod_rows)
        rr, yr, qr = oracle.scale_residual_nss_fp8(inp["x"], inp["residual"],
                                                   inp["bias"] if with_bias else None,
                                                   inp["gate"], inp["scale"], inp["shift"], s,
                                                   mod_rows=mod_rows)
        what = f"random {case}: {rows}x{cols}/{mod_rows} bias={with_bias} in_place={in_place}"
        assert np.array_equal(rg, rr), what
        check_ln(yg, qg, yr, qr, s, what)
        y = G.Guarded((rows, cols), torch.bfloat16)
        fq().bias_mul_add(G.dev_bf16(inp["x"]), G.dev_bf16(inp["bias"]),
                          G.dev_bf16(inp["gate"][0]), G.dev_bf16(inp["residual"]), y=y.tensor)
        torch.cuda.synchronize()
        assert y.intact()
        assert np.array_equal(G.host_u16(y.tensor), oracle.bias_mul_add(
            inp["x"], inp["bias"], inp["gate"][0], inp["residual"])), what


def test_random_sweep_token_cat_fp8_and_nvfp4():
    rng = np.random.default_rng(2028)
    for case in range(16):
        rows = int(rng.integers(1, 400))
        a_cols, m_cols = 64 * int(rng.integers(1, 100)), 64 * int(rng.integers(1, 300))
        inp = W.token_cat_inputs(rows, a_cols, m_cols, seed=3000 + case)
        s = _random_scale(rng)
        assert np.array_equal(run_token_cat(inp["a"], inp["m"], s),
                              oracle.token_cat_fp8(inp["a"], inp["m"], s)), f"fp8 random {case}"
        g = float(np.float32(10 ** rng.uniform(-3, 6)))
        check_nvfp4(inp["a"], inp["m"], g, f"nvfp4 random {case}: {rows}x{a_cols}+{m_cols} g={g}")


def test_random_sweep_qkv_epilogue():
    rng = np.random.default_rng(2029)
    for case in range(12):
        heads = int(rng.integers(1, 71))   # both the ring (<= 64 heads) and the per-token kernel
        tt, it = int(rng.integers(0, 40)), int(rng.integers(0, 80))
        if tt + it == 0:
            it = 1
        d = W.qkv_inputs(tt, it, heads, seed=4000 + case, extra_cols=16 * int(rng.integers(0, 4)))
        d["txt"]["eps"] = float(rng.choice([1e-6, 1e-5]))
        check_qkv(d, heads, f"random {case}: {tt}+{it}x{heads}")
