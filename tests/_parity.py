"""Shared helpers of the GPU parity tests: tolerances and comparisons.

Bars (stated for the path, float64 oracle as reference):
  fp32 inputs:  max |gpu - oracle| <= 1e-4
  bf16 inputs:  max |gpu - oracle| <= 2e-2 and mean |gpu - oracle| <= 2e-3
                (over all outputs, zero rows included)
  rows with no admissible key: exact zeros on both sides; lse = -inf
  lse (natural log, fp32 on the GPU), on finite rows:
                max |diff| <= tol * max(1, max |lse_oracle|), tol = 1e-3 for
                16-bit inputs and 1e-5 for fp32.  The bar is relative to the
                lse's magnitude because its error is: the hardware tanh of the
                softcapped 16-bit path carries a relative error of about 2^-11
                into every capped logit (about 2.5e-3 of a logit of 5), and
                fp32 rounding of m + log2(l) grows with |lse|.
"""
import torch

BF16_MAX = 2e-2
BF16_MEAN = 2e-3
F32_MAX = 1e-4


def check_out(got: torch.Tensor, ref: torch.Tensor, dtype, what=""):
    g = got.detach().to("cpu", torch.float64).reshape(ref.shape)
    assert torch.isfinite(g).all(), f"{what}: non-finite output"
    err = (g - ref).abs()
    mx, mean = err.max().item(), err.mean().item()
    if dtype == torch.float32:
        assert mx <= F32_MAX, f"{what}: max abs err {mx:.3e} > {F32_MAX}"
    else:
        assert mx <= BF16_MAX, f"{what}: max abs err {mx:.3e} > {BF16_MAX}"
        assert mean <= BF16_MEAN, f"{what}: mean abs err {mean:.3e} > {BF16_MEAN}"
    zero = (ref == 0).all(dim=-1)
    if zero.any():
        assert (g[zero] == 0).all(), f"{what}: fully-masked rows are not exact zeros"
    return mx, mean


def check_lse(got: torch.Tensor, ref: torch.Tensor, dtype, what=""):
    g = got.detach().to("cpu", torch.float64).reshape(ref.shape)
    fin = torch.isfinite(ref)
    assert torch.equal(torch.isneginf(g), torch.isneginf(ref)), f"{what}: -inf lse rows differ"
    tol = 1e-5 if dtype == torch.float32 else 1e-3
    if fin.any():
        d = (g[fin] - ref[fin]).abs().max().item()
        assert d <= tol * max(1.0, ref[fin].abs().max().item()), f"{what}: lse err {d:.3e}"
