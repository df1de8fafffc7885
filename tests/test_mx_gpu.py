"""GPU parity of the MXFP8 and NVFP4 weight paths against the oracle.

The kernel decodes the codes to BF16 exactly (E4M3 * 2^k and E2M1 * E4M3 are
representable in BF16 for these inputs) and applies the NVFP4 tensor scale to
the FP32 sums, so the acceptance rule is the BF16 one.
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


def _run(sg, fmt, M, N, K, seed, rows=None):
    A, w1, w2 = si.make_mx(M, N, K, seed, fmt)
    Ad = A.to(DEV)
    if fmt == "mxfp8":
        Y = sg.swiglu_fused_mxfp8(Ad, w1[0].to(DEV), w1[1].to(DEV), w2[0].to(DEV), w2[1].to(DEV))
        o1, o2 = (w1[0].numpy(), w1[1].numpy()), (w2[0].numpy(), w2[1].numpy())
    else:
        g1 = torch.tensor([w1[2]], dtype=torch.float32, device=DEV)
        g2 = torch.tensor([w2[2]], dtype=torch.float32, device=DEV)
        Y = sg.swiglu_fused_nvfp4(Ad, w1[0].to(DEV), w1[1].to(DEV), g1, w2[0].to(DEV), w2[1].to(DEV), g2)
        # the kernel reads the scales as binary32; the oracle takes the same values
        o1 = (w1[0].numpy(), w1[1].numpy(), float(np.float32(w1[2])))
        o2 = (w2[0].numpy(), w2[1].numpy(), float(np.float32(w2[2])))
    rc, detail = sg.swiglu_device_status()
    assert rc == sg.OK, (sg.status_string(rc), detail)
    ref = oracle.swiglu_mx(si.bits_u16(A), fmt, o1, o2, rows=rows)
    got = Y.double().cpu().numpy()
    if rows is not None:
        got = got[rows]
    oracle.assert_parity(got, ref, f"{fmt} {M}x{N}x{K}")


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("shape", [(1, 64, 64), (7, 96, 128), (63, 288, 384), (128, 4864, 896),
                                   (200, 160, 512), (65, 4864, 896),
                                   # wide weight matrices: the 128-column one-CTA kernel
                                   (37, 9760, 256), (130, 9856, 192),
                                   # two 128-row blocks per CTA, the last CTA's second
                                   # block wholly below the matrix
                                   (300, 9760, 256)],
                         ids=lambda s: "x".join(map(str, s)))
def test_mx_shapes(sg, fmt, shape):
    M, N, K = shape
    _run(sg, fmt, M, N, K, seed=M + N + K)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("M", [128, 256])  # the wide kernel with one and with two row blocks
def test_mx_7b_shape_sampled(sg, fmt, M):
    N, K = 18944, 3584
    _run(sg, fmt, M, N, K, seed=2, rows=si.sample_rows(M, 128, 32, seed=2))


# ---- MXFP8 codes K-major ([N, K], the transpose), decoded into tensor memory ----------------

def _run_mxfp8_kmajor(sg, M, N, K, seed, rows=None):
    A, w1, w2 = si.make_mx(M, N, K, seed, "mxfp8")
    C1k = w1[0].t().contiguous().to(DEV)
    C2k = w2[0].t().contiguous().to(DEV)
    Y = sg.swiglu_fused_mxfp8_kmajor(A.to(DEV), C1k, w1[1].to(DEV), C2k, w2[1].to(DEV))
    rc, detail = sg.swiglu_device_status()
    assert rc == sg.OK, (sg.status_string(rc), detail)
    o1, o2 = (w1[0].numpy(), w1[1].numpy()), (w2[0].numpy(), w2[1].numpy())
    ref = oracle.swiglu_mx(si.bits_u16(A), "mxfp8", o1, o2, rows=rows)
    got = Y.double().cpu().numpy()
    if rows is not None:
        got = got[rows]
    oracle.assert_parity(got, ref, f"mxfp8 k-major {M}x{N}x{K}")


@pytest.mark.parametrize("shape", [(1, 64, 64), (7, 96, 128), (63, 288, 384), (64, 4864, 896),
                                   (65, 4896, 896), (128, 1152, 448),
                                   # several 128-token passes, the last one ragged
                                   (300, 640, 256), (129, 256, 128),
                                   # ragged last column block (9760 = 76 x 128 + 32)
                                   (100, 9760, 256)],
                         ids=lambda s: "x".join(map(str, s)))
def test_mxfp8_kmajor_shapes(sg, shape):
    M, N, K = shape
    _run_mxfp8_kmajor(sg, M, N, K, seed=7 * M + N + K)


@pytest.mark.parametrize("M", [64, 128])
def test_mxfp8_kmajor_7b_shape_sampled(sg, M):
    N, K = 18944, 3584
    _run_mxfp8_kmajor(sg, M, N, K, seed=8, rows=si.sample_rows(M, 64, 24, seed=8))


def test_mxfp8_kmajor_argument_errors(sg):
    lib = sg.lib()
    A = torch.zeros(4, 128, dtype=torch.bfloat16, device=DEV)
    Ck = torch.zeros(64, 128, dtype=torch.uint8, device=DEV)
    S = torch.zeros(4, 64, dtype=torch.uint8, device=DEV)
    Y = torch.empty(4, 64, dtype=torch.bfloat16, device=DEV)
    p = [t.data_ptr() for t in (A, Ck, S, Ck, S, Y)]
    f = lib.swiglu_fused_mxfp8_kmajor
    assert f(*p, 4, 64, 96, None) == sg.ERR_UNSUPPORTED                        # K not a multiple of 64
    assert f(*p, 4, 48, 128, None) == sg.ERR_MISALIGNED                        # N not a multiple of 32
    assert f(*p[:5], A.data_ptr(), 4, 64, 128, None) == sg.ERR_INVALID_ARG     # Y overlaps A
    assert f(p[0], None, *p[2:], 4, 64, 128, None) == sg.ERR_INVALID_ARG       # missing codes
    assert f(*p, 0, 64, 128, None) == sg.OK
    Y.fill_(3.0)                                                               # K = 0: Y = 0
    assert f(*p, 4, 64, 0, None) == sg.OK
    torch.cuda.synchronize()
    assert torch.all(Y == 0)


# ---- NVFP4 codes in the K-major layout, decoded into tensor memory --------------------------

def _run_nvfp4_kmajor(sg, M, N, K, seed, rows=None):
    A, w1, w2 = si.make_mx(M, N, K, seed, "nvfp4")
    # E2M1 codes share INT4's [K, N/2] nibble layout: the INT4 packer serves both
    C1k = sg.swiglu_pack_w4_kmajor(w1[0].to(DEV))
    C2k = sg.swiglu_pack_w4_kmajor(w2[0].to(DEV))
    g1 = torch.tensor([w1[2]], dtype=torch.float32, device=DEV)
    g2 = torch.tensor([w2[2]], dtype=torch.float32, device=DEV)
    Y = sg.swiglu_fused_nvfp4_kmajor(A.to(DEV), C1k, w1[1].to(DEV), g1, C2k, w2[1].to(DEV), g2)
    rc, detail = sg.swiglu_device_status()
    assert rc == sg.OK, (sg.status_string(rc), detail)
    assert np.array_equal(C2k.cpu().numpy(), oracle.pack_w4_kmajor(w2[0].numpy()))
    o1 = (w1[0].numpy(), w1[1].numpy(), float(np.float32(w1[2])))
    o2 = (w2[0].numpy(), w2[1].numpy(), float(np.float32(w2[2])))
    ref = oracle.swiglu_mx(si.bits_u16(A), "nvfp4", o1, o2, rows=rows)
    got = Y.double().cpu().numpy()
    if rows is not None:
        got = got[rows]
    oracle.assert_parity(got, ref, f"nvfp4 k-major {M}x{N}x{K}")


@pytest.mark.parametrize("shape", [(1, 64, 64), (7, 96, 128), (63, 288, 384), (64, 4864, 896),
                                   (65, 4896, 896), (128, 1152, 448),
                                   # several 128-token passes, the last one ragged
                                   (300, 640, 256), (129, 256, 128),
                                   # ragged last column block (9760 = 76 x 128 + 32)
                                   (100, 9760, 256)],
                         ids=lambda s: "x".join(map(str, s)))
def test_nvfp4_kmajor_shapes(sg, shape):
    M, N, K = shape
    _run_nvfp4_kmajor(sg, M, N, K, seed=5 * M + N + K)


@pytest.mark.parametrize("M", [64, 128])
def test_nvfp4_kmajor_7b_shape_sampled(sg, M):
    N, K = 18944, 3584
    _run_nvfp4_kmajor(sg, M, N, K, seed=6, rows=si.sample_rows(M, 64, 24, seed=6))


def test_nvfp4_kmajor_argument_errors(sg):
    lib = sg.lib()
    A = torch.zeros(4, 128, dtype=torch.bfloat16, device=DEV)
    Ck = torch.zeros(64, 64, dtype=torch.uint8, device=DEV)
    S = torch.zeros(8, 64, dtype=torch.uint8, device=DEV)
    g = torch.ones(1, device=DEV)
    Y = torch.empty(4, 64, dtype=torch.bfloat16, device=DEV)
    p = [A.data_ptr(), Ck.data_ptr(), S.data_ptr(), g.data_ptr(), Ck.data_ptr(), S.data_ptr(), g.data_ptr(),
         Y.data_ptr()]
    f = lib.swiglu_fused_nvfp4_kmajor
    assert f(*p, 4, 64, 96, None) == sg.ERR_UNSUPPORTED                        # K not a multiple of 64
    assert f(*p, 4, 48, 128, None) == sg.ERR_MISALIGNED                        # N not a multiple of 32
    assert f(*p[:3], None, *p[4:], 4, 64, 128, None) == sg.ERR_INVALID_ARG     # missing tensor scale
    assert f(*p[:7], A.data_ptr(), 4, 64, 128, None) == sg.ERR_INVALID_ARG     # Y overlaps A
    assert f(*p, 0, 64, 128, None) == sg.OK
    Y.fill_(3.0)                                                               # K = 0: Y = 0
    assert f(*p, 4, 64, 0, None) == sg.OK
    torch.cuda.synchronize()
    assert torch.all(Y == 0)


def test_mx_argument_errors(sg):
    lib = sg.lib()
    A = torch.zeros(4, 128, dtype=torch.bfloat16, device=DEV)
    C = torch.zeros(128, 64, dtype=torch.uint8, device=DEV)
    S = torch.zeros(8, 64, dtype=torch.uint8, device=DEV)
    g = torch.ones(1, device=DEV)
    Y = torch.empty(4, 64, dtype=torch.bfloat16, device=DEV)
    pm = [A.data_ptr(), C.data_ptr(), S.data_ptr(), C.data_ptr(), S.data_ptr(), Y.data_ptr()]
    assert lib.swiglu_fused_mxfp8(*pm, 4, 64, 96, None) == sg.ERR_UNSUPPORTED      # K not a multiple of 64
    assert lib.swiglu_fused_mxfp8(*pm, 4, 48, 128, None) == sg.ERR_MISALIGNED      # N not a multiple of 32
    pn = [A.data_ptr(), C.data_ptr(), S.data_ptr(), None, C.data_ptr(), S.data_ptr(), g.data_ptr(), Y.data_ptr()]
    assert lib.swiglu_fused_nvfp4(*pn, 4, 64, 128, None) == sg.ERR_INVALID_ARG     # missing tensor scale
    torch.cuda.synchronize()
