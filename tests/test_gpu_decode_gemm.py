"""Batch-invariant decode GEMM at a fixed token width (GPU).

"ninfer" issue 80: decode GEMMs that pick their kernel or schedule from the
step's token count t change reduction order between compositions (the issue
measures boundaries at t = 5, 8, 17, 24, 32 on its shapes); at a fixed width
T_pad with padded activations the schedule is one for every t <= T_pad.
Parity: the CUDA path against the fp64 oracle within a rounding bound derived
from the arithmetic (fp32 accumulation over K, one bf16 rounding). Invariance:
the page's own experiment -- row 0 fixed, t = 1..T_pad real rows, the rest
NaN padding -- must leave y[0] bit-identical.
"""
import numpy as np
import pytest
import torch

import oracle.decode_gemm as dg
from helpers import to_store
from invariant_paged_kv_gb300 import build, pa

pytestmark = pytest.mark.gpu

# shapes (N, K) the issue lists for its W8 decode path
SHAPES = [(1024, 5120), (6144, 5120), (5120, 6144), (5120, 17408), (34816, 5120)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    pa.load()


def _inputs(T_pad, N, K, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn(T_pad, K, generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g, device="cuda") / K ** 0.5).to(torch.bfloat16)
    return x, w


def _check(y, x, w, rows=None):
    """|y - ref| <= K 2^-24 sum|x w| (fp32 accumulation) + 2^-8 |ref| (bf16 rounding)."""
    xs, ws = to_store(x), to_store(w)
    if rows is not None:
        ws = ws[rows]
        y = y[:, torch.as_tensor(rows, device=y.device)]
    ref = dg.linear(xs, ws)
    bound = x.shape[1] * 2.0 ** -24 * dg.abs_sum(xs, ws) + 2.0 ** -8 * np.abs(ref)
    got = y.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert (err <= bound).all(), float((err - bound).max())
    return float(err.max())


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("T_pad", [32, 64, 128])
def test_parity(N, K, T_pad):
    x, w = _inputs(T_pad, N, K, N + K + T_pad)
    y = torch.full((T_pad, N), float("nan"), device="cuda", dtype=torch.bfloat16)
    st = pa.new_status()
    pa.decode_gemm(x, w, y, status=st)
    assert pa.read_status(st) == 0
    _check(y, x, w)


def test_vocab_head_sampled():
    """The issue's vocabulary head [248320 x 5120] (2.5 GB of weights): all
    tokens, sampled weight rows (first and last tiles, random rows)."""
    N, K, T_pad = 248320, 5120, 64
    x, w = _inputs(T_pad, N, K, 9)
    y = torch.empty(T_pad, N, device="cuda", dtype=torch.bfloat16)
    pa.decode_gemm(x, w, y)
    rng = np.random.default_rng(0)
    rows = sorted(set(list(range(128)) + list(range(N - 128, N)) +
                      list(rng.integers(0, N, size=256))))
    _check(y, x, w, rows)


@pytest.mark.parametrize("N,K", [(1024, 5120), (6144, 5120), (34816, 5120)])
def test_row_bits_independent_of_token_count(N, K):
    """Splits: 20, 7 and 2 for these shapes (pa_decode_gemm_splits)."""
    T_pad = 64
    x, w = _inputs(T_pad, N, K, 77)
    y = torch.empty(T_pad, N, device="cuda", dtype=torch.bfloat16)
    ref = None
    for t in range(1, T_pad + 1):
        xt = x.clone()
        xt[t:] = float("nan")  # padding rows
        pa.decode_gemm(xt, w, y)
        row0 = y[0].clone()
        if ref is None:
            ref = row0
        assert torch.equal(row0.view(torch.int16), ref.view(torch.int16)), t
        assert torch.isfinite(y[:t].float()).all()
    _check(y, x, w)  # the last call had every row real


def test_padding_content_is_irrelevant():
    N, K, T_pad = 6144, 5120, 64
    x, w = _inputs(T_pad, N, K, 5)
    y1 = torch.empty(T_pad, N, device="cuda", dtype=torch.bfloat16)
    y2 = torch.empty_like(y1)
    pa.decode_gemm(x, w, y1)
    x2 = x.clone()
    x2[17:] = torch.randn(T_pad - 17, K, device="cuda").to(torch.bfloat16) * 1e4
    pa.decode_gemm(x2, w, y2)
    assert torch.equal(y1[:17].view(torch.int16), y2[:17].view(torch.int16))
