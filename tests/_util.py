"""Shared helpers of the test suite (comparison bar, sampling)."""
import numpy as np

# Parity bar for bf16 in / fp32 accumulate against the fp64 oracle.
MAX_ABS = 2e-2
REL_L2 = 1e-2


def to_f64(t):
    return t.detach().float().cpu().double().numpy()


def compare(got, ref, max_abs=MAX_ABS, rel_l2=REL_L2, what=""):
    """Element-wise bar: max |got - ref| <= max_abs and ||got-ref|| / ||ref|| <= rel_l2."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    d = np.abs(got - ref)
    nr = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / (nr if nr > 0 else 1.0)
    assert d.max() <= max_abs and rel <= rel_l2, (
        f"{what}: max|err|={d.max():.4e} (bar {max_abs}) relL2={rel:.4e} (bar {rel_l2}) "
        f"max|ref|={np.abs(ref).max():.3f} at {np.unravel_index(np.argmax(d), d.shape)}")
    return float(d.max()), float(rel)


def sample_points(T, H, W, n_random, seed):
    """(t, y, x) samples covering every boundary class (first frames, last
    frame, edge rows/columns, corners) plus uniform random interior ones."""
    rng = np.random.default_rng(seed)
    ts = sorted({0, min(1, T - 1), T - 1})
    ys = sorted({0, H - 1, H // 2})
    xs = sorted({0, W - 1, W // 2})
    pts = {(t, y, x) for t in ts for y in ys for x in xs}
    for _ in range(n_random):
        pts.add((int(rng.integers(T)), int(rng.integers(H)), int(rng.integers(W))))
    return sorted(pts)
