"""Helpers for the GPU parity tests: place a case on the device, run it
through the C ABI inside guard bands, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import dense_gemm_linear_gb300 as dgl
import oracle

# canaries: a NaN bit pattern no kernel produces from finite inputs
CANARY_BF16 = 0x7FC1
CANARY_F32 = 0x7FC00001
DEV = "cuda"


def to_device(case):
    """Device tensors of a case: (A, B, sa, sb)."""
    if case.dtype == "bf16":
        A = torch.from_numpy(case.A.view(np.int16)).view(torch.bfloat16).to(DEV)
        B = torch.from_numpy(case.B.view(np.int16)).view(torch.bfloat16).to(DEV)
        return A, B, None, None
    A = torch.from_numpy(case.A).view(torch.float8_e4m3fn).to(DEV)
    B = torch.from_numpy(case.B).view(torch.float8_e4m3fn).to(DEV)
    return A, B, torch.from_numpy(case.sa).to(DEV), torch.from_numpy(case.sb).to(DEV)


def canary_buffer(rows, cols, out):
    if out == "f32":
        return torch.full((rows, cols), CANARY_F32, dtype=torch.int32, device=DEV).view(torch.float32)
    return torch.full((rows, cols), CANARY_BF16, dtype=torch.int16, device=DEV).view(torch.bfloat16)


def run(case, *, guard_rows=0, pad_cols=0, plan=None, dev_ops=None, stream=None, base_offset=0):
    """Run the case through the C ABI.  C is a (m + guard_rows) x (n + pad_cols)
    buffer prefilled with canaries, starting base_offset elements into its
    allocation; returns (device C buffer, canaries_intact)."""
    A, B, sa, sb = dev_ops if dev_ops is not None else to_device(case)
    m, n, K = case.m, case.n, case.K
    rows, ldc = m + guard_rows, n + pad_cols
    if base_offset:
        flat = canary_buffer(1, rows * ldc + base_offset, case.out).view(-1)
        lead = flat[:base_offset]
        Cbuf = flat[base_offset:].view(rows, ldc)
    else:
        lead = None
        Cbuf = canary_buffer(rows, ldc, case.out)
    out_dtype = dgl.OUT_F32 if case.out == "f32" else dgl.OUT_BF16
    s = (stream or torch.cuda.current_stream()).cuda_stream
    if plan is not None:
        st = dgl.dgl_gemm_planned(dgl.DTYPE_BF16 if case.dtype == "bf16" else dgl.DTYPE_E4M3,
                                  A.data_ptr(), B.data_ptr(),
                                  sa.data_ptr() if sa is not None else None,
                                  sb.data_ptr() if sb is not None else None,
                                  Cbuf.data_ptr(), rows, ldc, K, m, n, out_dtype, plan, s)
    elif case.dtype == "bf16":
        st = dgl.dgl_gemm_bf16(A.data_ptr(), B.data_ptr(), Cbuf.data_ptr(), rows, ldc, K, m, n, out_dtype, s)
    else:
        st = dgl.dgl_gemm_fp8(A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(), Cbuf.data_ptr(),
                              rows, ldc, K, m, n, out_dtype, s)
    assert st == dgl.DGL_OK, dgl.status_string(st)
    st = dgl.dgl_device_status(s)
    assert st == dgl.DGL_OK, f"device status: {dgl.status_string(st)}"
    bits = Cbuf.view(torch.int32) if case.out == "f32" else Cbuf.view(torch.int16)
    canary = CANARY_F32 if case.out == "f32" else CANARY_BF16
    intact = bool((bits[m:, :] == canary).all().item()) and bool((bits[:m, n:] == canary).all().item())
    if lead is not None:
        lb = lead.view(torch.int32) if case.out == "f32" else lead.view(torch.int16)
        intact = intact and bool((lb == canary).all().item())
    return Cbuf, intact


def host_valid(case, Cbuf):
    """The valid region of a device C buffer as float64 numpy."""
    return Cbuf[:case.m, :case.n].double().cpu().numpy()


def oracle_dtype(case):
    return oracle.BF16 if case.dtype == "bf16" else oracle.E4M3


def tolerance(case, ref, S):
    """|C - C_ref| <= 1e-4 * S + 1e-6 (fp32 out); plus 1e-2 |C_ref| for bf16 out."""
    rel = 1e-2 if case.out == "bf16" else 0.0
    return rel * np.abs(ref) + 1e-4 * S + 1e-6


def assert_close_full(case, C):
    ref, S = oracle.gemm(oracle_dtype(case), case.A, case.B, case.sa, case.sb)
    _assert_within(case, C, ref, S, None)
    return ref


def _assert_within(case, got, ref, S, where):
    assert np.isfinite(got).all(), f"{case.name}: non-finite output"
    err = np.abs(got - ref)
    bound = tolerance(case, ref, S)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(tuple(int(v) for v in i), float(got[tuple(i)]), float(ref[tuple(i)])) for i in idx]
        raise AssertionError(f"{case.name}: {int(bad.sum())} of {bad.size} out of tolerance "
                             f"(max err {float(err.max()):.3e}); first {detail} at {where}")


def assert_exact(case, C):
    """Integer-valued inputs: the fp32 output equals the exact sum; bf16 output
    equals the exact sum rounded to nearest even."""
    ref, _ = oracle.gemm(oracle_dtype(case), case.A, case.B, case.sa, case.sb)
    if case.out == "f32":
        want = ref.astype(np.float32).astype(np.float64)
        assert np.array_equal(want, ref), "reference not exact in fp32 (test setup)"
        mism = C != ref
    else:
        want_bits = oracle.round_bf16(ref)
        got_bits = torch.from_numpy(C.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        mism = got_bits != want_bits
    if mism.any():
        idx = np.argwhere(mism)[:5]
        raise AssertionError(f"{case.name}: {int(mism.sum())} elements differ from the exact result; "
                             f"first {[(tuple(map(int, i)), float(C[tuple(i)]), float(ref[tuple(i)])) for i in idx]}")


def sample_points(case, tile_m, tile_n, seed, count=4096):
    """Seeded sample of the valid region plus full tiles at every ragged edge."""
    rng = np.random.default_rng(seed + 99)
    m, n = case.m, case.n
    rows = [rng.integers(0, m, size=count)]
    cols = [rng.integers(0, n, size=count)]
    tm, tn = min(tile_m, m), min(tile_n, n)
    blocks = [(m - tm, n - tn), (m - tm, 0), (0, n - tn), (0, 0)]
    for r0, c0 in blocks:
        rr, cc = np.meshgrid(np.arange(r0, r0 + tm), np.arange(c0, c0 + tn), indexing="ij")
        rows.append(rr.ravel())
        cols.append(cc.ravel())
    return np.concatenate(rows), np.concatenate(cols)


def assert_close_sampled(case, Cbuf, tile_m=256, tile_n=256, seed=0):
    """Check a seeded sample plus full edge tiles of the device buffer Cbuf."""
    rows, cols = sample_points(case, tile_m, tile_n, seed)
    ref, S = oracle.gemm_points(oracle_dtype(case), case.A, case.B, rows, cols, case.sa, case.sb)
    r_t = torch.from_numpy(rows).to(Cbuf.device)
    c_t = torch.from_numpy(cols).to(Cbuf.device)
    got = Cbuf[r_t, c_t].double().cpu().numpy()
    _assert_within(case, got, ref, S, "sampled points")
