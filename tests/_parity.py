"""Shared helpers of the GPU parity tests (host <-> device marshalling and
the comparison rules)."""
import numpy as np

# Attention outputs (bf16): max-abs and mean-abs bounds of the parity bar.
ATTN_MAX_ABS = 1e-2
ATTN_MEAN_ABS = 1e-3
# lse = ln(sum_j exp(l_j)): the readout sums the probabilities rounded to
# bf16, the operands of its PV product (relative error <= 2^-9 each), so the
# sum is within a relative 2^-9 of the exact one and lse within 2^-9 (plus
# the fp32 summation error).
LSE_ABS = 2.0 ** -9 + 1e-5
# Top-k sets: an index may differ only when its oracle score is within this
# relative distance of the oracle's k-th score (fp32 accumulation order on
# the tensor cores differs from the fp64 oracle).
NEAR_TIE_REL = 1e-5


def bf16_dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)) \
        .view(torch.bfloat16).to(device)


def f32_dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def bf16_host(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check_topk(gpu_idx, oracle_idx, oracle_scores, k, log=None):
    """Sets must match except near-ties; both lists ascending with -1 tail.
    Returns the number of near-tie differences (logged to ``log``)."""
    g = np.asarray(gpu_idx)
    o = np.asarray(oracle_idx)
    n_valid = int((o >= 0).sum())
    assert int((g >= 0).sum()) == n_valid, "different k_eff"
    assert np.all(g[n_valid:] == -1)
    assert np.all(np.diff(g[:n_valid]) > 0), "not strictly ascending"
    if n_valid == 0:
        return 0
    diff = set(g[:n_valid].tolist()) ^ set(o[:n_valid].tolist())
    if not diff:
        return 0
    kth = np.sort(np.asarray(oracle_scores, np.float64))[::-1][n_valid - 1]
    for i in diff:
        assert 0 <= i < len(oracle_scores)
        rel = abs(oracle_scores[i] - kth) / max(abs(kth), 1e-30)
        assert rel <= NEAR_TIE_REL, f"index {i}: score {oracle_scores[i]} vs k-th {kth}"
        if log is not None:
            log.append((int(i), float(oracle_scores[i]), float(kth)))
    return len(diff)


def check_lse(gpu_lse, oracle_lse, where=""):
    g = np.asarray(gpu_lse, np.float64)
    o = np.asarray(oracle_lse, np.float64)
    fin = np.isfinite(o)
    assert np.array_equal(np.isfinite(g), fin), where
    err = np.abs(g[fin] - o[fin])
    assert err.size == 0 or err.max() <= LSE_ABS, f"{where} lse max err {err.max()}"


def check_attn(gpu_out_bf16_bits, oracle_out_f64, strict=False):
    """bf16 GPU output against the fp64 oracle.  Max-abs 1e-2 and mean-abs
    1e-3; where |o| >= 2.56 a single bf16 rounding step already exceeds 1e-2
    (half an ulp is 2^-8 |o|), so there the per-element bound is one bf16 ulp,
    2^-7 |o|.  ``strict`` applies the flat 1e-2 everywhere (workload
    distributions, whose outputs stay below that magnitude)."""
    from csa2_synth import bf16_bits_to_f32
    g = bf16_bits_to_f32(gpu_out_bf16_bits).astype(np.float64)
    ref = np.asarray(oracle_out_f64, np.float64)
    err = np.abs(g - ref)
    assert np.all(np.isfinite(g))
    tol = ATTN_MAX_ABS if strict else np.maximum(ATTN_MAX_ABS, 2.0 ** -7 * np.abs(ref))
    bad = err > tol
    assert not bad.any(), f"max abs err {err.max()} at |o| = {np.abs(ref)[bad].max()}"
    assert err.mean() <= ATTN_MEAN_ABS, f"mean abs err {err.mean()}"
    return float(err.max()), float(err.mean())
