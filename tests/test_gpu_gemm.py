"""The product engine in isolation (mt_debug_gemm): every operand layout the
update uses - K-major and MN-major A and B, ragged rows (expert segments of
ragged_mm) and ragged reductions (expert weight gradients) - on the
tensor-core path (bf16 operands) and on the CUDA-core path of the fp32 model
(the same bf16-valued inputs held in fp32), against a float64 product."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TOL = 2e-3          # relative L2: fp32 accumulation of bf16 products in a different order


def _arena():
    from adamw_persistent_sm_gb300 import binding as B
    arena = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    assert B.mt_arena_init(arena.data_ptr(), arena.numel()) == B.MT_OK
    return arena


def _run(A, a_mn, Bm, b_mn, M, N, K, rag=0, offs=None, nseg=0, use_tc=1, out_shape=None):
    from adamw_persistent_sm_gb300 import binding as B
    arena = _arena()
    if not (use_tc & 1):                 # the CUDA-core engine is the fp32 model's
        A, Bm = A.float(), Bm.float()
    C = torch.full(out_shape or (M, N), float("nan"), dtype=torch.float32, device="cuda")
    prec = B.MT_PREC_BF16 if A.dtype == torch.bfloat16 else B.MT_PREC_FP32
    st = B.mt_debug_gemm(A.data_ptr(), a_mn, Bm.data_ptr(), b_mn, C.data_ptr(), M, N, K, rag,
                         offs.data_ptr() if offs is not None else 0, nseg, prec, use_tc,
                         arena.data_ptr(), arena.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == B.MT_OK, B.status_string(st)
    out = B.mt_read_outputs(arena.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert out.status == B.MT_OK, (B.status_string(out.status), out.error_site)
    return C


def _rel(a, b):
    a = a.double().cpu()
    b = b.double().cpu()
    return float((a - b).norm() / b.norm())


@pytest.mark.parametrize("use_tc", [1, 0])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
def test_dense_layouts(use_tc, a_mn, b_mn):
    torch.manual_seed(0)
    M, N, K = 384, 512, 448
    a = torch.randn(M, K, device="cuda").bfloat16()
    b = torch.randn(N, K, device="cuda").bfloat16()
    A = a.t().contiguous() if a_mn else a
    Bm = b.t().contiguous() if b_mn else b
    C = _run(A, a_mn, Bm, b_mn, M, N, K, use_tc=use_tc)
    ref = a.double() @ b.double().t()
    assert _rel(C, ref) < TOL


@pytest.mark.parametrize("use_tc", [1, 0])
@pytest.mark.parametrize("b_mn", [0, 1])
def test_ragged_rows(use_tc, b_mn):
    """Rows in expert segments padded to 128; segment e uses weight e."""
    torch.manual_seed(1)
    nseg, N, K = 4, 256, 192
    counts = [128, 0, 256, 128]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(offs[-1]) + 128                      # rows past offs[-1] stay untouched
    a = torch.randn(M, K, device="cuda").bfloat16()
    w = torch.randn(nseg, N, K, device="cuda").bfloat16()
    Bm = w.transpose(1, 2).contiguous() if b_mn else w
    C = _run(a, 0, Bm, b_mn, M, N, K, rag=1, offs=torch.as_tensor(offs).cuda(), nseg=nseg, use_tc=use_tc)
    for e in range(nseg):
        r0, r1 = offs[e], offs[e + 1]
        if r1 > r0:
            assert _rel(C[r0:r1], a[r0:r1].double() @ w[e].double().t()) < TOL
    assert torch.isnan(C[offs[-1]:]).all()


@pytest.mark.parametrize("use_tc", [1, 0])
def test_ragged_reduction(use_tc):
    """Weight-gradient shape: C[e] = A_e^T B_e over segment e's rows; an
    empty segment gives zeros."""
    torch.manual_seed(2)
    nseg, M, N = 3, 256, 512
    counts = [256, 0, 384]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    K = int(offs[-1])
    a = torch.randn(K, M, device="cuda").bfloat16()      # [rows, M]: MN-major A
    b = torch.randn(K, N, device="cuda").bfloat16()      # [rows, N]: MN-major B
    C = _run(a, 1, b, 1, M, N, K, rag=2, offs=torch.as_tensor(offs).cuda(), nseg=nseg, use_tc=use_tc,
             out_shape=(nseg, M, N))
    for e in range(nseg):
        r0, r1 = offs[e], offs[e + 1]
        if r1 > r0:
            assert _rel(C[e], a[r0:r1].double().t() @ b[r0:r1].double()) < TOL
        else:
            assert torch.all(C[e] == 0)


def test_fp32_simt_exact():
    torch.manual_seed(3)
    M, N, K = 100, 70, 33                        # ragged tails on every side
    a = torch.randn(M, K, device="cuda")
    b = torch.randn(K, N, device="cuda")
    C = _run(a, 0, b, 1, M, N, K, use_tc=0)
    assert _rel(C, a.double() @ b.double()) < 1e-6


@pytest.mark.parametrize("bf16_out", [0, 1])
@pytest.mark.parametrize("rag", [0, 1])
def test_bulk_store_epilogue(bf16_out, rag):
    """C written by the bulk-store epilogue (swizzled shared-memory boxes and
    bulk tensor stores, the path of the update's products) equals the plain
    stores of the same product bit for bit, and matches the float64 product."""
    from adamw_persistent_sm_gb300 import binding as B
    torch.manual_seed(4)
    N, K = 512, 320
    offs = None
    nseg = 0
    if rag:
        counts = [256, 0, 128]
        nseg = len(counts)
        offs_np = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        offs = torch.as_tensor(offs_np).cuda()
        M = int(offs_np[-1])
        w = torch.randn(nseg, N, K, device="cuda").bfloat16()
    else:
        M = 384
        w = torch.randn(N, K, device="cuda").bfloat16()
    a = torch.randn(M, K, device="cuda").bfloat16()
    mode = 1 | (bf16_out << 1)
    plain = _run(a, 0, w, 0, M, N, K, rag=rag, offs=offs, nseg=nseg, use_tc=mode)
    bulk = _run(a, 0, w, 0, M, N, K, rag=rag, offs=offs, nseg=nseg, use_tc=mode | 8)
    if bf16_out:
        # bf16 C occupies the first M*N*2 bytes of the buffer
        plain = plain.view(torch.bfloat16).reshape(-1)[:M * N].reshape(M, N).float()
        bulk = bulk.view(torch.bfloat16).reshape(-1)[:M * N].reshape(M, N).float()
    assert torch.equal(plain, bulk)
    if rag:
        ref = torch.cat([a[offs_np[e]:offs_np[e + 1]].double() @ w[e].double().t() for e in range(nseg)])
    else:
        ref = a.double() @ w.double().t()
    assert _rel(bulk, ref) < (1e-2 if bf16_out else TOL)


def test_bf16_operands_have_no_cuda_core_path():
    from adamw_persistent_sm_gb300 import binding as B
    arena = _arena()
    a = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(256, 64, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(128, 256, dtype=torch.float32, device="cuda")
    st = B.mt_debug_gemm(a.data_ptr(), 0, b.data_ptr(), 0, c.data_ptr(), 128, 256, 64, 0, 0, 0,
                         B.MT_PREC_BF16, 0, arena.data_ptr(), arena.numel(),
                         torch.cuda.current_stream().cuda_stream)
    assert st == B.MT_ERR_UNSUPPORTED
