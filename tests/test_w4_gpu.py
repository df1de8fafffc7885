"""GPU parity of the INT4-weight path against the oracle.

Both sides use the same weights, BF16(q * s) (the kernel decodes them in
shared memory, the oracle in double then rounds to BF16 identically), so the
acceptance rule is the BF16 one: FP32 accumulation and the BF16 rounding of Y
are the only differences.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_inputs as si

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def sg():
    import __graft_entry__
    __graft_entry__.build()
    import swiglu_gemm_transformer_gb300 as m
    m.lib()
    return m


def _run(sg, M, N, K, G, seed, rows=None):
    A, (W1q, S1), (W2q, S2) = si.make_w4(M, N, K, seed, G)
    Y = sg.swiglu_fused_w4(A.to(DEV), W1q.to(DEV), S1.to(DEV), W2q.to(DEV), S2.to(DEV), group=G)
    rc, detail = sg.swiglu_device_status()
    assert rc == sg.OK, (sg.status_string(rc), detail)
    ref = oracle.swiglu_w4(si.bits_u16(A), W1q.numpy(), si.bits_u16(S1), W2q.numpy(),
                           si.bits_u16(S2), G, rows=rows)
    got = Y.double().cpu().numpy()
    if rows is not None:
        got = got[rows]
    oracle.assert_parity(got, ref, f"w4 {M}x{N}x{K} G={G}")


@pytest.mark.parametrize("shape", [(1, 64, 128, 128), (7, 96, 256, 64), (63, 288, 384, 128),
                                   (128, 4864, 896, 128), (200, 160, 512, 128), (384, 320, 640, 64),
                                   (65, 4864, 896, 128),
                                   # wide weight matrices: the 128-column one-CTA kernel, with
                                   # a ragged last tile (9760 = 76 x 128 + 32) and ragged M
                                   (37, 9760, 256, 128), (130, 9856, 192, 64),
                                   # two 128-row blocks per CTA, the last CTA's second
                                   # block wholly below the matrix
                                   (300, 9760, 256, 128)],
                         ids=lambda s: "x".join(map(str, s)))
def test_w4_shapes(sg, shape):
    M, N, K, G = shape
    _run(sg, M, N, K, G, seed=M + N + K)


@pytest.mark.parametrize("M", [128, 256])  # the wide kernel with one and with two row blocks
def test_w4_7b_shape_sampled(sg, M):
    N, K = 18944, 3584
    _run(sg, M, N, K, 128, seed=2, rows=si.sample_rows(M, 128, 32, seed=2))


def test_w4_read_only_mode(sg):
    sg.swiglu_set_weights_read_only(True)
    try:
        _run(sg, 128, 4864, 896, 128, seed=5)
        _run(sg, 63, 288, 384, 128, seed=6)
    finally:
        sg.swiglu_set_weights_read_only(False)


def test_w4_argument_errors(sg):
    lib = sg.lib()
    A = torch.zeros(4, 128, dtype=torch.bfloat16, device=DEV)
    Wq = torch.zeros(128, 32, dtype=torch.uint8, device=DEV)
    S = torch.zeros(1, 64, dtype=torch.bfloat16, device=DEV)
    Y = torch.empty(4, 64, dtype=torch.bfloat16, device=DEV)
    p = [t.data_ptr() for t in (A, Wq, S, Wq, S, Y)]
    assert lib.swiglu_fused_w4(*p, 4, 64, 128, 100, None) == sg.ERR_UNSUPPORTED   # group not a multiple of 64
    assert lib.swiglu_fused_w4(*p, 4, 64, 128, 256, None) == sg.ERR_UNSUPPORTED   # group does not divide K
    assert lib.swiglu_fused_w4(*p, 4, 48, 128, 128, None) == sg.ERR_MISALIGNED    # N not a multiple of 32
    assert lib.swiglu_fused_w4(*p, -1, 64, 128, 128, None) == sg.ERR_INVALID_ARG
    # K = 0: every product is zero
    Y.fill_(3.0)
    assert lib.swiglu_fused_w4(*p, 4, 64, 0, 128, None) == sg.OK
    torch.cuda.synchronize()
    assert torch.all(Y == 0)


# ---- K-major codes decoded into tensor memory (swiglu_fused_w4_kmajor) -----------------------

def _run_kmajor(sg, M, N, K, G, seed, rows=None):
    A, (W1q, S1), (W2q, S2) = si.make_w4(M, N, K, seed, G)
    W1k = sg.swiglu_pack_w4_kmajor(W1q.to(DEV))
    W2k = sg.swiglu_pack_w4_kmajor(W2q.to(DEV))
    Y = sg.swiglu_fused_w4_kmajor(A.to(DEV), W1k, S1.to(DEV), W2k, S2.to(DEV), group=G)
    rc, detail = sg.swiglu_device_status()
    assert rc == sg.OK, (sg.status_string(rc), detail)
    # the packer against the oracle's arrangement, byte for byte
    assert np.array_equal(W1k.cpu().numpy(), oracle.pack_w4_kmajor(W1q.numpy()))
    ref = oracle.swiglu_w4(si.bits_u16(A), W1q.numpy(), si.bits_u16(S1), W2q.numpy(),
                           si.bits_u16(S2), G, rows=rows)
    got = Y.double().cpu().numpy()
    if rows is not None:
        got = got[rows]
    oracle.assert_parity(got, ref, f"w4 k-major {M}x{N}x{K} G={G}")


@pytest.mark.parametrize("shape", [(1, 128, 64, 64), (17, 256, 192, 64), (64, 4864, 896, 128),
                                   (65, 4896, 896, 128), (128, 1152, 448, 64),
                                   # several 128-token passes, the last one ragged
                                   (300, 640, 256, 128), (129, 256, 128, 128),
                                   # ragged last column block (9760 = 76 x 128 + 32), one group
                                   (100, 9760, 256, 256)],
                         ids=lambda s: "x".join(map(str, s)))
def test_w4_kmajor_shapes(sg, shape):
    M, N, K, G = shape
    _run_kmajor(sg, M, N, K, G, seed=3 * M + N + K)


@pytest.mark.parametrize("M", [64, 128])
def test_w4_kmajor_7b_shape_sampled(sg, M):
    N, K = 18944, 3584
    _run_kmajor(sg, M, N, K, 128, seed=4, rows=si.sample_rows(M, 64, 24, seed=4))


def test_w4_kmajor_argument_errors(sg):
    lib = sg.lib()
    A = torch.zeros(4, 128, dtype=torch.bfloat16, device=DEV)
    Wk = torch.zeros(64, 64, dtype=torch.uint8, device=DEV)
    S = torch.zeros(1, 64, dtype=torch.bfloat16, device=DEV)
    Y = torch.empty(4, 64, dtype=torch.bfloat16, device=DEV)
    p = [t.data_ptr() for t in (A, Wk, S, Wk, S, Y)]
    assert lib.swiglu_fused_w4_kmajor(*p, 4, 64, 128, 100, None) == sg.ERR_UNSUPPORTED
    assert lib.swiglu_fused_w4_kmajor(*p, 4, 48, 128, 128, None) == sg.ERR_MISALIGNED
    assert lib.swiglu_fused_w4_kmajor(p[0], p[1], p[2], p[3], p[4], p[0], 4, 64, 128, 128, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_fused_w4_kmajor(*p, 0, 64, 128, 128, None) == sg.OK
    Y.fill_(3.0)                                                               # K = 0: Y = 0
    assert lib.swiglu_fused_w4_kmajor(*p, 4, 64, 0, 128, None) == sg.OK
    torch.cuda.synchronize()
    assert torch.all(Y == 0)
    assert lib.swiglu_pack_w4_kmajor(p[1], p[1], 128, 64, None) == sg.ERR_INVALID_ARG  # overlap
    assert lib.swiglu_pack_w4_kmajor(p[1], Y.data_ptr(), 12, 64, None) == sg.ERR_MISALIGNED
