"""Parity checks shared by the GPU tests: the CUDA result against the CPU
oracle, with the tolerances the workload statement fixes.

GEMV outputs:  |gpu - ref| <= 1e-3 * sum_j |w_ij x_j| + 1e-6, NaN == NaN.
FFN / MoE outputs: the oracle's first-order propagation of that bound
through SwiGLU, the routing weights and the down product (oracle.c,
orc_moe_ffn).  Routing: expert indices bit-exact, in rank order, for every
token whose top k+1 logits are separated by more than AMBIGUITY times the
router's max_e sum_j |R_ej x_j|.  For the rest ("ambiguous" tokens) the
GPU's route must be a valid top-k within that margin; if it equals the
oracle's, the outputs are compared as usual, otherwise the two forwards
took different (equally valid) experts and only the route is checked.

AMBIGUITY: the router kernel sums each logit as 16 sequential FMAs per
thread, 5 shuffle levels and 4 partial sums, so its f32 error is at most
about 25 * 2^-24 * sum_j |R_ej x_j| ~ 1.5e-6 of that scale; two logits can
swap only if they lie within twice that.  1e-5 leaves a 3x margin.
"""
import numpy as np

AMBIGUITY = 1e-5


class ParityError(AssertionError):
    pass


def check_close(got, want, tol, what="output"):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    tol = np.broadcast_to(np.asarray(tol, dtype=np.float64), want.shape)
    if got.shape != want.shape:
        raise ParityError(f"{what}: shape {got.shape} != {want.shape}")
    nan_w = np.isnan(want)
    if not np.array_equal(np.isnan(got), nan_w):
        bad = np.flatnonzero(np.isnan(got) != nan_w)[:5]
        raise ParityError(f"{what}: NaN mismatch at {bad.tolist()}")
    inf_w = np.isinf(want)
    if np.any(~np.isfinite(got[~nan_w]) != inf_w[~nan_w]):
        raise ParityError(f"{what}: Inf mismatch")
    ok = np.isfinite(want)
    err = np.abs(got[ok] - want[ok])
    lim = tol[ok]
    if np.any(err > lim):
        i = int(np.argmax(err - lim))
        flat = np.flatnonzero(ok)[i]
        raise ParityError(
            f"{what}: |err| {err[i]:.3e} > tol {lim[i]:.3e} at {flat} "
            f"(got {got.flat[flat]!r}, want {want.flat[flat]!r}); "
            f"{int(np.sum(err > lim))} of {err.size} outside")
    return float(np.max(err / lim)) if err.size else 0.0


def gemv_tol(sabs):
    return 1e-3 * np.asarray(sabs) + 1e-6


def check_gemv(y_gpu, y_ref, sabs, what="y"):
    return check_close(y_gpu, y_ref, gemv_tol(sabs), what)


def route_is_valid(idx, logits, scale, k, margin=AMBIGUITY):
    """idx is a top-k of `logits` in rank order, up to ties within margin*scale."""
    idx = np.asarray(idx)
    if len(set(idx.tolist())) != k or np.any(idx < 0) or np.any(idx >= logits.size):
        return False
    eps = 2 * margin * scale
    kth = np.sort(logits)[::-1][k - 1]
    if np.any(logits[idx] < kth - eps):
        return False
    return bool(np.all(np.diff(logits[idx]) <= eps))


def check_moe(out_gpu, idx_gpu, w_gpu, ref, what="moe"):
    """ref: dict from oracle.moe_ffn.  Returns the number of ambiguous tokens
    whose (valid) route differs from the oracle's."""
    out_gpu = np.asarray(out_gpu).reshape(ref["out"].shape)
    idx_gpu = np.asarray(idx_gpu).reshape(ref["idx"].shape)
    k = idx_gpu.shape[1]
    amb = ref["gap"] <= AMBIGUITY
    same = np.array([np.array_equal(idx_gpu[t], ref["idx"][t]) for t in range(len(amb))])
    for t in np.flatnonzero(~same):
        if not amb[t]:
            raise ParityError(f"{what}: token {t} routed to {idx_gpu[t].tolist()}, "
                              f"oracle {ref['idx'][t].tolist()}")
        if not route_is_valid(idx_gpu[t], ref["logits"][t], ref["lscale"][t], k):
            raise ParityError(f"{what}: token {t} route {idx_gpu[t].tolist()} is not a top-{k} "
                              f"of the oracle logits within the margin")
    if w_gpu is not None:
        w_gpu = np.asarray(w_gpu).reshape(ref["w"].shape)
        check_close(w_gpu[same], ref["w"][same], 1e-5 * np.abs(ref["w"][same]) + 1e-6,
                    f"{what} routing weights")
    check_close(out_gpu[same], ref["out"][same], ref["tol"][same], f"{what} residual")
    return int(np.sum(~same))
