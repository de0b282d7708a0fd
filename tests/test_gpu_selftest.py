"""GPU check of the tcgen05 / TMA building blocks: one 128 x N x 128 tile
D = A B^T on the tensor cores, operands staged by threads (hand-written
128-byte swizzle) or by TMA (hardware swizzle), against a torch fp32 matmul."""
import ctypes
import os

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def selftest():
    from kda_chunked_prefill_02_gb300 import build
    build.build()
    lib = ctypes.CDLL(build.SELFTEST_LIB)
    lib.kda_selftest_umma.restype = ctypes.c_int
    lib.kda_selftest_umma.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 2 + [ctypes.c_void_p] * 2
    return lib


@pytest.mark.parametrize("use_tma", [0, 1])
@pytest.mark.parametrize("N", [32, 64, 96, 256])
def test_umma_tile(selftest, N, use_tma):
    g = torch.Generator(device="cpu").manual_seed(N + use_tma)
    A = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(N, 128, generator=g).to(torch.bfloat16).cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = selftest.kda_selftest_umma(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, use_tma,
                                    status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and status.item() == 0
    ref = A.float() @ B.float().T
    torch.testing.assert_close(D, ref, atol=2e-3, rtol=1e-4)


@pytest.mark.parametrize("N", [32, 64, 128, 256])
def test_umma_tile_b_mn_major(selftest, N):
    """B stored MN-major (128-byte swizzle, atoms along N 1024 B apart, 8-row K
    groups max(N/64, 1) KB apart): the layout of the prep kernel's [K e^Gam | V]
    (N = 256) and of the state pass's S and V_new operands (N = 32)."""
    f = selftest.kda_selftest_umma_mn
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 2 + [ctypes.c_void_p] * 2
    g = torch.Generator(device="cpu").manual_seed(100 + N)
    A = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(N, 128, generator=g).to(torch.bfloat16).cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert f(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, 0, status.data_ptr(),
             torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert status.item() == 0
    torch.testing.assert_close(D, A.float() @ B.float().T, atol=2e-3, rtol=1e-4)


def test_umma_tile_b_mn_major_sw64(selftest):
    """N = 32 B operand stored MN-major with the 64-byte swizzle (64-byte rows,
    8-row groups 512 B apart): the state pass's S and V operands."""
    f = selftest.kda_selftest_umma_mn64
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 5
    g = torch.Generator(device="cpu").manual_seed(77)
    A = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(32, 128, generator=g).to(torch.bfloat16).cuda()
    D = torch.full((128, 32), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert f(A.data_ptr(), B.data_ptr(), D.data_ptr(), status.data_ptr(),
             torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert status.item() == 0
    torch.testing.assert_close(D, A.float() @ B.float().T, atol=2e-3, rtol=1e-4)


@pytest.mark.parametrize("N", [32, 128])
def test_umma_tile_a_from_tmem(selftest, N):
    """A operand (128 x 128 bf16) read by the MMA from TMEM, packed two bf16 per
    32-bit column (row m in lane m), B K-major SW128 in shared memory."""
    f = selftest.kda_selftest_umma_tmem_a
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] + [ctypes.c_void_p] * 2
    g = torch.Generator(device="cpu").manual_seed(300 + N)
    A = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(N, 128, generator=g).to(torch.bfloat16).cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert f(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, status.data_ptr(),
             torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert status.item() == 0
    torch.testing.assert_close(D, A.float() @ B.float().T, atol=2e-3, rtol=1e-4)


@pytest.mark.parametrize("N", [128, 192])
def test_umma_tile_a_from_tmem_fp16(selftest, N):
    """The same with fp16 A and B (both operands of one product share the type):
    the whole-chain state kernel's V_new^T [Kt ; Aqk]^T (N = 192)."""
    f = selftest.kda_selftest_umma_tmem_a_typed
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 2 + [ctypes.c_void_p] * 2
    g = torch.Generator(device="cpu").manual_seed(310 + N)
    A = torch.randn(128, 128, generator=g).to(torch.float16).cuda()
    B = torch.randn(N, 128, generator=g).to(torch.float16).cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert f(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, 1, status.data_ptr(),
             torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert status.item() == 0
    torch.testing.assert_close(D, A.float() @ B.float().T, atol=2e-3, rtol=1e-4)


def test_umma_tile_b_mn_major_fp16(selftest):
    """fp16 A (K-major) and B (MN-major, N = 32): the slab state kernel's
    Kt V_new and Aqk V_new."""
    f = selftest.kda_selftest_umma_mn
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 2 + [ctypes.c_void_p] * 2
    g = torch.Generator(device="cpu").manual_seed(150)
    A = torch.randn(128, 128, generator=g).to(torch.float16).cuda()
    B = torch.randn(32, 128, generator=g).to(torch.float16).cuda()
    D = torch.full((128, 32), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert f(A.data_ptr(), B.data_ptr(), D.data_ptr(), 32, 2, status.data_ptr(),
             torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert status.item() == 0
    torch.testing.assert_close(D, A.float() @ B.float().T, atol=2e-3, rtol=1e-4)


@pytest.mark.parametrize("N", [32, 64])
def test_umma_tile_a_and_b_mn_major(selftest, N):
    """A stored MN-major too (A^T as [K rows][M contiguous], two 64-row atoms
    1 KB apart): the form of prep's U^T = V^T T'^T, whose A operand is the V
    half of the [K e^Gam | V] operand."""
    f = selftest.kda_selftest_umma_mn
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 2 + [ctypes.c_void_p] * 2
    g = torch.Generator(device="cpu").manual_seed(170 + N)
    A = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(N, 128, generator=g).to(torch.bfloat16).cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert f(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, 4, status.data_ptr(),
             torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert status.item() == 0
    torch.testing.assert_close(D, A.float() @ B.float().T, atol=2e-3, rtol=1e-4)


def test_mma_rate_probe_runs(selftest):
    """The MMA throughput probe (back-to-back tcgen05.mma of one shape, timed
    with clock64 on the issuing thread) completes and reports a positive time."""
    f = selftest.kda_selftest_mma_rate
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    cyc = torch.zeros(2, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for mode in (0, 4):
        assert f(mode, 8, cyc.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        assert status.item() == 0
        issue, total = cyc.tolist()
        assert 0 < issue <= total


def test_tf32_rounding_matches_the_conversion_instruction(selftest):
    """to_tf32 (two integer operations: add half a unit of the 13 dropped
    mantissa bits, then drop them) equals cvt.rna.tf32.f32 bit for bit on
    finite values: random values over the whole exponent range, exact ties of
    both signs, ties that carry into the exponent, subnormals and zeros."""
    f = selftest.kda_selftest_tf32_round
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_void_p]
    gen = torch.Generator().manual_seed(11)
    bits = torch.randint(0, 2 ** 31, (1 << 20,), generator=gen, dtype=torch.int64)
    bits = bits | (torch.randint(0, 2, bits.shape, generator=gen) << 31)
    bits = bits[((bits >> 23) & 0xFF) != 0xFF]                      # finite only
    # and finite once rounded (nothing within half a tf32 unit of the top)
    bits = bits[(((bits >> 23) & 0xFF) != 0xFE) | ((bits & 0x7FFFFF) < 0x7FF000)]
    mant = torch.randint(0, 1 << 10, (4096,), generator=gen, dtype=torch.int64)
    expo = torch.randint(1, 254, (4096,), generator=gen, dtype=torch.int64)
    ties = (expo << 23) | (mant << 13) | 0x1000                    # exactly half way
    carry = (expo << 23) | (0x3FF << 13) | torch.randint(0x1000, 0x2000, (4096,), generator=gen)
    special = torch.tensor([0, 1, 0x1000, 0x1FFF, 0x7FFFFF, 0x800000, 0x7F7FEFFF], dtype=torch.int64)
    extra = torch.cat([ties, carry, special])
    bits = torch.cat([bits, extra, extra | (1 << 31)])
    # the 32-bit patterns as int32 (two's complement), viewed as fp32
    x = (((bits & 0xFFFFFFFF) + (1 << 31)) % (1 << 32) - (1 << 31)).to(torch.int32).view(torch.float32).cuda()
    n = x.numel()
    fast = torch.empty(n, dtype=torch.int32, device="cuda")
    ref = torch.empty(n, dtype=torch.int32, device="cuda")
    assert f(x.data_ptr(), fast.data_ptr(), ref.data_ptr(), n, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    bad = (fast != ref).nonzero().flatten()
    assert bad.numel() == 0, (x[bad[:8]].tolist(), fast[bad[:8]].tolist(), ref[bad[:8]].tolist())


def _tf32(x):
    """fp32 -> the tf32 value the tensor core uses (the low 13 mantissa bits
    dropped)."""
    b = x.contiguous().view(torch.int32) & ~0x1FFF
    return b.view(torch.float32)


@pytest.mark.parametrize("a_mn,b_mn,N,K", [(0, 0, 32, 128), (0, 0, 16, 128), (0, 0, 128, 16),
                                           (0, 0, 128, 8), (0, 0, 64, 64), (2, 0, 32, 128),
                                           (2, 0, 128, 128)])
def test_umma_tf32_operand_forms(selftest, a_mn, b_mn, N, K):
    """tcgen05 kind::tf32 with K-major operands (128-byte swizzle, fp32
    elements) in shared memory, or A (a_mn = 2) in TMEM, one element per
    column, row m in lane m: the forms of the tensor-core verify kernel's two
    products (S^T [W; Q']^T with S^T in TMEM: N = 32, K = 128; V_new^T Kt_a^T:
    N = 128, K = 8 or 16), against a matmul of the tf32-rounded operands.
    (tf32 operands in shared memory must be K-major: an MN-major tf32 operand
    gave zeros on GB300.)"""
    f = selftest.kda_selftest_umma_tf32
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 2
    g = torch.Generator(device="cpu").manual_seed(900 + N + K + 2 * a_mn + b_mn)
    A = torch.randn(128, K, generator=g).cuda()
    B = torch.randn(N, K, generator=g).cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert f(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, K, a_mn, b_mn, status.data_ptr(),
             torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert status.item() == 0
    ref = (_tf32(A).double() @ _tf32(B).double().T).float()
    torch.testing.assert_close(D, ref, atol=1e-4, rtol=1e-5)
