"""Tolerances and comparison helpers shared by the GPU parity tests.

The bars: attention outputs with bf16 inputs within max-abs 2e-2 and
mean-abs 2e-3 of the fp64 oracle; with fp32 inputs within 1e-4; LSE within
1e-3 absolute; append and gather bit-exact."""
import numpy as np
import torch

BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
F32_MAX_ABS = 1e-4
LSE_ABS = 1e-3


def to_np(t):
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def assert_out_close(gpu, ref, fp32_inputs=False, what="out"):
    g, r = to_np(gpu), np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - r)
    if fp32_inputs:
        assert err.max() <= F32_MAX_ABS, f"{what}: max abs err {err.max():.3g} > {F32_MAX_ABS}"
    else:
        assert err.max() <= BF16_MAX_ABS, f"{what}: max abs err {err.max():.3g} > {BF16_MAX_ABS}"
        assert err.mean() <= BF16_MEAN_ABS, f"{what}: mean abs err {err.mean():.3g} > {BF16_MEAN_ABS}"
    return err.max(), err.mean()


def assert_lse_close(gpu, ref, what="lse"):
    g, r = to_np(gpu), np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    both_inf = np.isneginf(g) & np.isneginf(r)
    assert np.array_equal(np.isneginf(g), np.isneginf(r)), f"{what}: -inf pattern differs"
    with np.errstate(invalid="ignore"):  # -inf - -inf where both are -inf, masked out
        err = np.abs(np.where(both_inf, 0.0, g - r))
    assert err.max() <= LSE_ABS, f"{what}: max abs err {err.max():.3g} > {LSE_ABS}"
    return err.max()


def sample_rows(B, H, P, n, seed):
    """Seeded query rows (flat ids (b*H + h)*P + i) that always include the
    first and last row of the first and last head and two rows late in the
    last head (where the last wave's query tiles sit), plus random ones."""
    rng = np.random.default_rng(seed)
    last = (B * H - 1) * P
    fixed = [0, P - 1, last, B * H * P - 1, last + (9 * P) // 10, last + (19 * P) // 20]
    rnd = rng.choice(B * H * P, size=max(0, n - len(fixed)), replace=False)
    return np.unique(np.concatenate([np.array(fixed), rnd]).astype(np.int64))
