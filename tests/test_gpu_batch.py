"""dgl_gemm_batch: independent GEMMs back to back on one stream, each kernel
after the first reading its operands while its predecessor still runs and
waiting for it only before writing C.  Checked against the oracle, and for
the two orderings the call promises: work enqueued before the batch is seen
by every item, and work enqueued after it sees every item's C.

Integer-valued inputs make every expected value exact (the same recipes as
the single-call tests), so a result computed from stale operands, or read
before its kernel finished, shows as a mismatch, not as a rounding difference.
"""
import numpy as np
import pytest
import torch

import dense_gemm_linear_gb300 as dgl
import oracle
from synthetic import make_case
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

DTYPE_ID = {"bf16": dgl.DTYPE_BF16, "fp8": dgl.DTYPE_E4M3, "w4a8": dgl.DTYPE_W4A8, "mxfp4": dgl.DTYPE_MXFP4}


def _ops(case):
    """Device operands (A, B, scale_a, scale_b) in the layouts the single calls take."""
    if case.dtype == "bf16":
        A, B, _, _ = gu.to_device(case)
        return A, B, None, None
    if case.dtype == "fp8":
        return gu.to_device(case)
    A = torch.from_numpy(case.A).to(gu.DEV)
    B = torch.from_numpy(case.B).to(gu.DEV)
    return A, B, torch.from_numpy(case.sa).to(gu.DEV), torch.from_numpy(case.sb).to(gu.DEV)


def _reference(case, rows=None):
    """Exact expected values (integer inputs), of all rows or of `rows`."""
    A = case.A if rows is None else case.A[rows]
    sa = case.sa if rows is None or case.sa is None else case.sa[rows]
    if case.dtype == "mxfp4":
        return oracle.mxfp4_gemm(A, case.B, sa, case.sb)[0]
    if case.dtype == "w4a8":
        return oracle.w4a8_gemm(A, case.B, sa, case.sb)[0]
    return oracle.gemm(oracle.BF16 if case.dtype == "bf16" else oracle.E4M3, A, case.B, sa, case.sb)[0]


def _exact(case, got, ref):
    if case.out == "f32":
        assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref), "test setup: reference not exact"
        mism = got != ref
    else:
        want = oracle.round_bf16(ref)
        have = torch.from_numpy(got.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        mism = have != want
    assert not mism.any(), f"{case.name}: {int(mism.sum())} of {mism.size} elements differ from the exact result"


class Item:
    """One batch item: its case, device operands and a canary-filled C with guard bands."""

    def __init__(self, case, guard_rows=2, pad_cols=3, ops=None, C=None):
        self.case = case
        self.ops = ops if ops is not None else _ops(case)
        rows, ldc = case.m + guard_rows, case.n + pad_cols
        self.C = C if C is not None else gu.canary_buffer(rows, ldc, case.out)
        self.rows, self.ldc = self.C.shape

    def desc(self):
        A, B, sa, sb = self.ops
        c = self.case
        return dict(dtype=DTYPE_ID[c.dtype], out_dtype=dgl.OUT_F32 if c.out == "f32" else dgl.OUT_BF16,
                    A=A.data_ptr(), B=B.data_ptr(), scale_a=sa.data_ptr() if sa is not None else None,
                    scale_b=sb.data_ptr() if sb is not None else None, C=self.C.data_ptr(),
                    M=self.rows, N=self.ldc, K=c.K, m_valid=c.m, n_valid=c.n)

    def check(self):
        c = self.case
        bits = self.C.view(torch.int32) if c.out == "f32" else self.C.view(torch.int16)
        canary = gu.CANARY_F32 if c.out == "f32" else gu.CANARY_BF16
        assert bool((bits[c.m:, :] == canary).all().item()) and bool((bits[:c.m, c.n:] == canary).all().item()), \
            f"{c.name}: wrote outside the valid region"
        _exact(c, self.C[:c.m, :c.n].double().cpu().numpy(), _reference(c))


def _batch(items, stream=None):
    s = (stream or torch.cuda.current_stream()).cuda_stream
    st = dgl.dgl_gemm_batch([it.desc() for it in items], s)
    assert st == dgl.DGL_OK, dgl.status_string(st)
    return s


def test_batch_every_path_exact():
    """Tile kernels (row staging, TMA store, f32 out), the decode kernel, E4M3,
    W4A8 and MXFP4 items in one batch; every C exact and inside its guard band."""
    cases = [make_case("bf16", 300, 517, 256, out="bf16", dist="int"),     # row staging
             make_case("bf16", 8, 1001, 640, out="bf16", dist="int"),      # decode
             make_case("fp8", 260, 384, 512, out="f32", dist="int"),
             make_case("fp8", 16, 700, 1024, out="bf16", dist="int"),      # decode, E4M3
             make_case("w4a8", 200, 300, 512, out="f32", dist="int"),
             make_case("mxfp4", 190, 260, 512, out="f32", dist="int"),
             make_case("bf16", 129, 257, 200, out="f32", dist="int"),
             make_case("bf16", 640, 768, 1024, out="bf16", dist="int")]    # several waves of tiles
    items = [Item(c) for c in cases]
    s = _batch(items)
    assert dgl.dgl_device_status(s) == dgl.DGL_OK
    for it in items:
        it.check()


def test_batch_empty_and_zero_k_items():
    """An empty item enqueues nothing (its C keeps its canaries); a K = 0 item
    writes zeros; the items around them are exact."""
    a = Item(make_case("bf16", 200, 300, 128, out="f32", dist="int"))
    b = Item(make_case("bf16", 64, 96, 64, out="f32", dist="int"))
    z = Item(make_case("bf16", 40, 50, 64, out="f32", dist="int"))
    c = Item(make_case("fp8", 150, 260, 256, out="bf16", dist="int"))
    descs = [a.desc(), dict(b.desc(), M=0, m_valid=0), dict(z.desc(), K=0), c.desc()]
    s = torch.cuda.current_stream().cuda_stream
    assert dgl.dgl_gemm_batch(descs, s) == dgl.DGL_OK
    assert dgl.dgl_device_status(s) == dgl.DGL_OK
    a.check()
    c.check()
    assert bool((b.C.view(torch.int32) == gu.CANARY_F32).all().item()), "the empty item wrote"
    assert bool((z.C[:40, :50] == 0).all().item()), "K = 0 writes zeros"
    assert dgl.dgl_gemm_batch([], s) == dgl.DGL_OK


def test_batch_invalid_item_enqueues_nothing():
    """A misaligned item anywhere in the batch: its status is returned before
    anything is enqueued, so the valid items' C keep their canaries."""
    a = Item(make_case("bf16", 200, 300, 128, out="f32", dist="int"))
    bad = Item(make_case("bf16", 64, 96, 64, out="f32", dist="int"))
    s = torch.cuda.current_stream().cuda_stream
    st = dgl.dgl_gemm_batch([a.desc(), dict(bad.desc(), K=60)], s)   # K * 2 bytes not a multiple of 16
    assert st == dgl.DGL_ERR_ALIGN
    st = dgl.dgl_gemm_batch([a.desc(), dict(bad.desc(), dtype=9)], s)
    assert st == dgl.DGL_ERR_ARG
    torch.cuda.synchronize()
    assert bool((a.C.view(torch.int32) == gu.CANARY_F32).all().item()), "an item was enqueued"


def test_batch_sees_work_enqueued_before_it():
    """The operands of every item are written on the stream right before the
    batch, behind a long GPU-side delay: each item (the later ones read their
    operands without waiting for their predecessor) must see the new values."""
    cases = [make_case("bf16", 256, 512, 512, out="f32", dist="int", seed=s) for s in range(4)]
    items = []
    fresh = []
    for c in cases:
        A, B, _, _ = _ops(c)
        A_buf = torch.zeros_like(A)
        items.append(Item(c, ops=(A_buf, B, None, None)))
        fresh.append((A_buf, A))
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)          # about a millisecond of GPU time before the copies land
        for A_buf, A in fresh:
            A_buf.copy_(A)
        _batch(items, stream)
    stream.synchronize()
    assert dgl.dgl_device_status(stream.cuda_stream) == dgl.DGL_OK
    for it in items:
        it.check()


def test_batch_work_after_it_sees_every_c():
    """A long first item and short later ones, then a copy of the first item's C
    on the same stream: the copy sees the finished C (each kernel of the batch
    completes only after the one before it)."""
    big = Item(make_case("bf16", 2048, 2048, 2048, out="f32", dist="int"), guard_rows=0, pad_cols=0)
    small = [Item(make_case("bf16", 8, 512, 256, out="f32", dist="int", seed=s)) for s in range(3)]
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        _batch([big] + small, stream)
        snap = big.C.clone()
    stream.synchronize()
    rows = np.array([0, 1, 511, 1024, 1535, 2047])
    ref = _reference(big.case, rows)
    _exact(big.case, snap[torch.from_numpy(rows).to(gu.DEV)].double().cpu().numpy(), ref)
    for it in small:
        it.check()


def test_batch_items_sharing_c_later_wins():
    """Two items writing the same C: the batch leaves the second one's result."""
    c1 = make_case("bf16", 300, 400, 256, out="f32", dist="int", seed=1)
    c2 = make_case("bf16", 300, 400, 256, out="f32", dist="int", seed=2)
    first = Item(c1)
    second = Item(c2, C=first.C)
    s = _batch([first, second])
    assert dgl.dgl_device_status(s) == dgl.DGL_OK
    second.check()


def test_batch_split_schedule_then_more_items():
    """An item the planner splits along K (a split-K tail through the stream's
    workspace) followed by items that start while it runs: all exact, twice."""
    case = make_case("bf16", 1200, 4800, 4096, out="f32", dist="int")
    p = dgl.dgl_plan(dgl.DTYPE_BF16, case.m, case.n, case.K, dgl.OUT_F32, num_sms=152)
    assert p.stream_k >= 2, "test setup: the planner should split this tail"
    big = Item(case)
    tail = [Item(make_case("bf16", 300, 300, 256, out="f32", dist="int", seed=s)) for s in range(2)]
    for _ in range(2):
        s = _batch([big] + tail)
        assert dgl.dgl_device_status(s) == dgl.DGL_OK
        rows = np.array([0, 255, 256, 1024, 1199])
        got = big.C[torch.from_numpy(rows).to(gu.DEV), :case.n].double().cpu().numpy()
        _exact(case, got, _reference(case, rows))
        for it in tail:
            it.check()


def test_batch_replayed_from_a_cuda_graph():
    """A batch captured into a CUDA graph and replayed after new operands were
    copied in: each replay computes from the new values."""
    cases = [make_case("bf16", 300, 517, 256, out="f32", dist="int", seed=s) for s in range(3)]
    alt = [make_case("bf16", 300, 517, 256, out="f32", dist="int", seed=10 + s) for s in range(3)]
    items = [Item(c) for c in cases]
    alt_A = [_ops(c)[0] for c in alt]
    # after the copies: the alternative A against each item's own B
    alt_ref = [oracle.gemm(oracle.BF16, a.A, c.B)[0] for a, c in zip(alt, cases)]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        _batch(items, stream)                # first use on this stream outside the capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        _batch(items, stream)
    for rnd in range(2):
        with torch.cuda.stream(stream):
            if rnd == 1:
                for it, A in zip(items, alt_A):
                    it.ops[0].copy_(A)
            g.replay()
        stream.synchronize()
        for i, (it, c) in enumerate(zip(items, cases)):
            got = it.C[:c.m, :c.n].double().cpu().numpy()
            _exact(c, got, _reference(c) if rnd == 0 else alt_ref[i])
