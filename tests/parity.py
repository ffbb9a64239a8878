"""Comparison rules between the CUDA path and the oracle.

* Expert ids are compared exactly for every token whose oracle logit gap
  between the k-th and (k+1)-th expert exceeds 1e-5 * (1 + |l_k|); the two
  sides rank fp32 logits summed in different orders, so closer gaps may
  legitimately flip.  Such tokens are counted and compared on output only.
* Routing weights: |w_gpu - w_oracle| <= 1e-5 (fp32 softmax vs fp64).
* Layer output (before the residual): max |y_gpu - y_oracle| <= 2e-2 * RMS(y_oracle),
  plus, when the GPU output carries the residual, the bf16 rounding of
  x + y (2^-8 * |x + y| elementwise).
"""
import numpy as np

TOL_REL_RMS = 2e-2
WEIGHT_ATOL = 1e-5


def bf16_to_f64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return (t.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return t.detach().float().cpu().numpy().astype(np.float64)


def margin_ok(logits: np.ndarray, k: int) -> np.ndarray:
    """Per token: True if the oracle's top-k set is separated by the margin."""
    srt = -np.sort(-logits.astype(np.float64), axis=-1)
    gap = srt[..., k - 1] - srt[..., k]
    return gap > 1e-5 * (1.0 + np.abs(srt[..., k - 1]))


def check_ids(ids_gpu, ref, k):
    """Exact ids where the margin holds; returns the number of near-tie tokens."""
    ok = margin_ok(ref["logits"], k)
    assert np.array_equal(np.asarray(ids_gpu)[ok], ref["ids"][ok]), "expert ids differ"
    return int((~ok).sum())


def check_weights(w_gpu, ref, ids_gpu):
    same = np.all(np.asarray(ids_gpu) == ref["ids"], axis=-1)
    if same.any():
        err = np.abs(np.asarray(w_gpu, np.float64)[same] - ref["w"][same]).max()
        assert err <= WEIGHT_ATOL, err


def check_output(y_gpu_bf16, y_ref, x_bf16=None):
    """y_ref: oracle fp64 [T, D] before the residual.  Returns max error / RMS."""
    g = bf16_to_f64(y_gpu_bf16)
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    if x_bf16 is None:
        err = np.abs(g - y_ref)
        tol = TOL_REL_RMS * rms
        assert err.max() <= tol, (err.max(), tol)
        return err.max() / rms
    x = bf16_to_f64(x_bf16)
    err = np.abs((g - x) - y_ref)
    tol = TOL_REL_RMS * rms + 2.0 ** -8 * np.abs(x + y_ref)
    assert np.all(err <= tol), (err.max(), rms)
    return err.max() / rms
