"""GPU parity of the down projection (Z = X W + R) and of the SwiGLU MLP block
(Z = BF16(SiLU(A W1) (.) (A W2)) W3 + R) against the oracle, element by
element (small shapes) or on sampled rows (Qwen-2.5 shapes).

The down projection uses the same acceptance rule as the fused projection.
The MLP block rounds Y to BF16 in between; the kernel rounds from an FP32
value and the oracle from the exact value, so near a rounding midpoint they
may pick neighbouring BF16 values (both correct roundings), and such a flip
moves every element of its row of Z by up to spacing * |W3[f,h]|.  The MLP
tests keep bound (1) on every element, and every significant element must
meet the 1 % rule (2) widened by its own slack: the sum over the Y elements
of its row that lie within the kernel's error of a midpoint of that
element's possible move (oracle.mlp_rounding_slack; the error model is in
oracle.check.bf16_rounding_slack).  No element is exempt.
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


def _residual(M, N, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(M, N, generator=g).to(torch.bfloat16)


def _status(sg):
    rc, detail = sg.swiglu_device_status()
    assert rc == sg.OK, f"device status {sg.status_string(rc)} detail {detail}"


# Few output tiles (small M) run the split-K cluster kernel: 64-column tiles
# over 4 CTAs for (63, 136, 200), (257, 392, 264), (300, 512, 1000) and
# (200, 896, 4864), over 8 for (128, 896, 4864), (100, 264, 520) and
# (64, 72, 4864) (a ragged last tile); 128-column tiles over 4 CTAs for
# (512, 896, 4864) and (128, 2600, 1000) (a ragged last tile), over 2 for
# (1024, 896, 4864); the others run the CTA-pair kernel.
@pytest.mark.parametrize("shape", [(1, 8, 8), (63, 136, 200), (257, 392, 264), (300, 512, 1000),
                                   (128, 896, 4864), (200, 896, 4864), (2048, 3584, 1024),
                                   (100, 264, 520), (64, 72, 4864), (512, 896, 4864),
                                   (128, 2600, 1000), (1024, 896, 4864)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("with_r", [False, True])
@pytest.mark.parametrize("with_ws", [True, False])
def test_linear(sg, shape, with_r, with_ws):
    M, N, K = shape
    X, W, _ = si.make_bf16(M, N, K, seed=M + N + K)
    R = _residual(M, N, 7) if with_r else None
    ws = None if with_ws else torch.empty(0, dtype=torch.uint8, device=DEV)
    Z = sg.swiglu_linear(X.to(DEV), W.to(DEV), R.to(DEV) if with_r else None, workspace=ws)
    _status(sg)
    ref = oracle.linear_bf16(si.bits_u16(X), si.bits_u16(W), si.bits_u16(R) if with_r else None)
    oracle.assert_parity(Z.float().cpu().numpy(), ref, f"linear {shape} r={with_r} ws={with_ws}")


@pytest.mark.parametrize("shape", [(130, 264, 136), (100, 264, 520)], ids=["pair", "cluster"])
def test_linear_in_place_residual(sg, shape):
    M, N, K = shape
    X, W, _ = si.make_bf16(M, N, K, seed=1)
    R = _residual(M, N, 2)
    Zd = R.clone().to(DEV)
    sg.swiglu_linear(X.to(DEV), W.to(DEV), Zd, Zd)
    _status(sg)
    ref = oracle.linear_bf16(si.bits_u16(X), si.bits_u16(W), si.bits_u16(R))
    oracle.assert_parity(Zd.float().cpu().numpy(), ref, f"in-place residual {shape}")


def test_linear_split_matches_unsplit(sg):
    M, N, K = 128, 896, 4864
    X, W, _ = si.make_bf16(M, N, K, seed=3)
    Xd, Wd = X.to(DEV), W.to(DEV)
    Z1 = sg.swiglu_linear(Xd, Wd)                                           # split K
    Z2 = sg.swiglu_linear(Xd, Wd, workspace=torch.empty(0, dtype=torch.uint8, device=DEV))
    _status(sg)
    # different summation orders: equal within the acceptance rule, not bitwise
    oracle.assert_parity(Z1.float().cpu().numpy(), Z2.double().cpu().numpy(), "split vs unsplit")


def test_linear_schedules_agree(sg):
    """The pair kernel's linear mode on more tiles than pairs fit (8 x 14 tiles
    of 256 x 256 here): the dynamic (cluster launch control) and static tile
    schedules give the same Z bit for bit, and both match the oracle."""
    M, N, K = 2048, 3584, 1024
    X, W, _ = si.make_bf16(M, N, K, seed=21)
    R = _residual(M, N, 22)
    out = {}
    try:
        for dyn in (1, 0):
            sg.swiglu_set_pair_schedule(dyn)
            out[dyn] = sg.swiglu_linear(X.to(DEV), W.to(DEV), R.to(DEV))
            _status(sg)
    finally:
        sg.swiglu_set_pair_schedule(1)
    assert torch.equal(out[0].view(torch.int16), out[1].view(torch.int16))
    rows = si.sample_rows(M, 256, 32, seed=21)
    ref = oracle.linear_bf16(si.bits_u16(X), si.bits_u16(W), si.bits_u16(R), rows=rows)
    oracle.assert_parity(out[1].float().cpu().numpy()[rows], ref, "linear, dynamic schedule")


MLP_CASES = [
    # (name, M, H, F, seed, residual)
    ("tiny", 7, 64, 136, 5, True),
    ("ragged", 200, 264, 520, 6, False),
    ("0.5b_m64", 64, 896, 4864, 0, True),
    ("0.5b_m128", 128, 896, 4864, 1, False),
    ("0.5b_m512", 512, 896, 4864, 1, True),
    ("0.5b_m2048", 2048, 896, 4864, 1, False),
    ("7b_m256", 256, 3584, 18944, 2, True),
]


@pytest.mark.parametrize("case", MLP_CASES, ids=lambda c: c[0])
def test_mlp(sg, case):
    name, M, H, F, seed, with_r = case
    A, W1, W2 = si.make_bf16(M, F, H, seed)
    W3 = si.make_bf16(1, H, F, seed + 100)[1]       # [F, H]
    R = _residual(M, H, seed) if with_r else None
    Z = sg.swiglu_mlp(A.to(DEV), W1.to(DEV), W2.to(DEV), W3.to(DEV), R.to(DEV) if with_r else None)
    _status(sg)
    rows = None if M <= 512 else si.sample_rows(M, 128, 32, seed)
    bits = [si.bits_u16(t) for t in (A, W1, W2, W3)]
    ref = oracle.mlp_bf16(*bits, si.bits_u16(R) if with_r else None, rows=rows)
    slack = oracle.mlp_rounding_slack(*bits, rows=rows)
    z = Z.float().cpu().numpy()
    oracle.assert_parity(z if rows is None else z[rows], ref, f"mlp {name}", sig_slack=slack)
