"""Tolerances of the GPU-vs-oracle comparisons.

The GPU keeps float32 inside each kernel and rounds to bf16 where a kernel
writes its output; the oracle is double throughout.  For one kernel fed
bit-identical bf16 inputs the only non-negligible difference is that final
rounding: at most half a unit in the 8-bit significand, i.e. 2^-8 * |ref|.
Float32 accumulation over K <= 57344 terms adds ~K * 2^-24 * sum|terms|,
covered by a small absolute term relative to the output's RMS.

Whole-model gates (logits in float32, hidden states in bf16) are the stated
max-abs bound 2e-2 (6e-2 for int8 weights); for the un-normalised residual
stream of deep stacks the bound is applied relative to max(1, |ref|) because one
bf16 unit there already exceeds 2e-2 once |x| > 4.
"""
import numpy as np
import torch

BF16_REL = 2.0 ** -8


def f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    import oracle
    return oracle.host_bits(t)


def assert_kernel_close(gpu, ref, rel=BF16_REL * 1.02, atol_rms=2e-4, what=""):
    g, r = f64(gpu), f64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    scale = max(1e-30, float(np.sqrt(np.mean(r * r))))
    bound = rel * np.abs(r) + atol_rms * scale
    err = np.abs(g - r)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {err.size} beyond bound; worst at {i}: "
                             f"gpu {g[i]!r} ref {r[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}")


def max_abs(a, b) -> float:
    return float(np.max(np.abs(f64(a) - f64(b))))


def assert_stream_close(gpu, ref, tol=2e-2, what=""):
    """Residual-stream gate: |gpu - ref| <= tol * max(1, |ref|, rms of ref's row).

    The path rounds the LayerNorm outputs, q / k / v, the attention output and
    the MLP intermediate to bf16 (relative error up to 2^-9 each); a block's
    contribution to the residual is a sum over K of such rounded values times
    weights, so its error grows with the row's scale, not with each element's
    own magnitude.  A restatement that rounds at the same points deviates from
    the float64 oracle by as much (7b1-width block, rms 2.7: max 4.2e-2), so
    elements small within a large row are bounded by the row's rms."""
    g, r = f64(gpu), f64(ref)
    err = np.abs(g - r)
    rms = np.sqrt(np.mean(r * r, axis=-1, keepdims=True)) if r.ndim else np.abs(r)
    bound = tol * np.maximum(np.maximum(1.0, np.abs(r)), rms)
    if (err > bound).any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: max|err| {err.max():.3e}; worst at {i}: gpu {g[i]} ref {r[i]}")


def greedy_agree(gpu_tokens, ref_logits, margin=0.1):
    """Tokens must equal the oracle's argmax wherever its top-2 margin > margin.
    Returns the number of rows checked."""
    ref = f64(ref_logits)
    gt = np.asarray(gpu_tokens).reshape(-1)
    top2 = np.sort(ref, axis=1)[:, -2:]
    checked = 0
    for b in range(ref.shape[0]):
        if top2[b, 1] - top2[b, 0] > margin:
            checked += 1
            assert int(gt[b]) == int(np.argmax(ref[b])), (b, int(gt[b]), int(np.argmax(ref[b])))
    return checked
