"""Shared helpers of the parity tests: the acceptance bound and GPU plumbing."""
import numpy as np

# Per-element acceptance: |y - y_ref| <= 1e-3 * sum_k |x_k w_kn| + 2^-10 * |y_ref|,
# y the GPU's FP16 output taken exactly to FP64, y_ref and the sum from the oracle.
REL_SUM = 1e-3
REL_OUT = 2.0 ** -10


# BF16 activations (derived, not stated by the target): BF16 keeps 8 significant
# bits, so the dequantised weight carries up to 2^-8 relative error where FP16's
# carries 2^-11. The FP16 bound allows about twice the weight rounding (1e-3 against
# 2^-11) for it and the FP32 accumulation; the same factor gives 2^-7 on the sum of
# |x*w|, and the output rounding to BF16 gives 2^-8 * |y_ref|.
REL_SUM_BF16 = 2.0 ** -7
REL_OUT_BF16 = 2.0 ** -8


def check_within(y_gpu, y_ref, absum, what="", rel_sum=REL_SUM, rel_out=REL_OUT):
    y = np.asarray(y_gpu, dtype=np.float64)
    bound = rel_sum * absum + rel_out * np.abs(y_ref)
    err = np.abs(y - y_ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.max(err / np.maximum(bound, 1e-300))
        raise AssertionError("%s: %d of %d outside the bound (worst err/bound %.3g); first at %s: gpu %s ref %s bound %s"
                             % (what, int(bad.sum()), bad.size, worst, idx.tolist(),
                                [y[tuple(i)] for i in idx], [y_ref[tuple(i)] for i in idx],
                                [bound[tuple(i)] for i in idx]))
    return float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0


# Fused epilogue y = act(z + b) + r: the GEMM term grows by the activation's largest
# slope (SiLU: 1.0998, ReLU and none: 1), plus FP32 rounding of the bias add, the
# activation and the residual add (2^-20 covers them with margin); the output
# rounding term is unchanged.
LIPSCHITZ_ACT = 1.1
REL_FP32_EPI = 2.0 ** -20


def check_within_fused(y_gpu, y_ref, z_ref, absum, bias_abs, resid_abs, what="", rel_sum=REL_SUM, rel_out=REL_OUT):
    y = np.asarray(y_gpu, dtype=np.float64)
    bound = (LIPSCHITZ_ACT * rel_sum * absum + rel_out * np.abs(y_ref)
             + REL_FP32_EPI * (np.abs(z_ref) + bias_abs + resid_abs + 1.0))
    err = np.abs(y - y_ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.max(err / np.maximum(bound, 1e-300))
        raise AssertionError("%s: %d of %d outside the bound (worst err/bound %.3g); first at %s: gpu %s ref %s"
                             % (what, int(bad.sum()), bad.size, worst, idx.tolist(),
                                [y[tuple(i)] for i in idx], [y_ref[tuple(i)] for i in idx]))
    return float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0


class forced_path:
    """Run a block with the library's dispatcher forced to one path (1: the CUDA-core
    kernel where it applies, 2: the tensor-core kernel); the previous setting is
    restored on exit."""

    def __init__(self, w, path):
        self.w, self.path = w, path

    def __enter__(self):
        self.prev = self.w.force_path(self.path)

    def __exit__(self, *exc):
        self.w.force_path(self.prev)
