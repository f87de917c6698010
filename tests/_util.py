"""Shared helpers for the GPU parity tests."""
import numpy as np
import torch

# Attention outputs on bf16 inputs: max-abs 2e-2 and mean-abs 2e-3 against the fp64 oracle.
ATOL_MAX = 2e-2
ATOL_MEAN = 2e-3


def assert_close(got: torch.Tensor, ref: np.ndarray, what: str = "", max_abs=ATOL_MAX, mean_abs=ATOL_MEAN):
    g = got.detach().float().cpu().double().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    assert err.max() <= max_abs, f"{what}: max abs err {err.max():.3e} > {max_abs}"
    assert err.mean() <= mean_abs, f"{what}: mean abs err {err.mean():.3e} > {mean_abs}"
    return float(err.max()), float(err.mean())


def sample_rows(B, H, N, n, seed=0, extra=()):
    """Flat query ids spread over (b, h) and the tile boundaries, plus the last row."""
    g = np.random.default_rng(seed)
    rows = set(int(r) for r in g.integers(0, B * H * N, size=n))
    for bh in (0, B * H - 1):
        for i in (0, 127, 128, 255, 256, N - 129, N - 2, N - 1):
            if 0 <= i < N:
                rows.add(bh * N + i)
    rows.update(extra)
    return np.array(sorted(rows), dtype=np.int64)


def check_device_status():
    import visual_autoregressive_next_var_b300 as V
    st = V.var_device_status(clear=True)
    assert st == 0, f"device status word: {st} ({V.var_status_string(st)})"


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """The oracle's own fp64 result stored as bf16 (round to nearest even through
    fp32), for chained stages whose next input is a stored bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).float().to(torch.bfloat16)


def csr_to_token_mask(sides, step, qbs, row_ptr, entries, sink_len):
    """Expand the library's block CSR into a [N, L] token mask (bool)."""
    sq = sides[step]
    nb = sq // qbs
    offs = np.cumsum([0] + [s * s for s in sides[: step + 1]])
    L = offs[-1]
    out = np.zeros((sq * sq, L), dtype=bool)
    for qb in range(nb * nb):
        by, bx = divmod(qb, nb)
        keys = np.zeros(L, dtype=bool)
        keys[:sink_len] = True
        for e in entries[row_ptr[qb]:row_ptr[qb + 1]]:
            sc, u, w = e >> 24, (e >> 12) & 0xFFF, e & 0xFFF
            s = sides[sc]
            for r in range(u * qbs, min(s, u * qbs + qbs)):
                c0, c1 = w * qbs, min(s, w * qbs + qbs)
                keys[offs[sc] + r * s + c0: offs[sc] + r * s + c1] = True
        for y in range(by * qbs, by * qbs + qbs):
            out[y * sq + bx * qbs: y * sq + bx * qbs + qbs] = keys
    return out
