"""Parity checks shared by the GPU tests: the CUDA result against the CPU
oracle, with the tolerances the workload statement fixes.

GEMV outputs:  |gpu - ref| <= 1e-3 * sum_j |w_ij x_j| + 1e-6, NaN == NaN.
FFN / MoE outputs: the oracle's first-order propagation of that bound
through SwiGLU, the routing weights and the down product (oracle.c,
orc_moe_ffn).  Routing: expert indices bit-exact, in rank order, for every
token whose top k+1 logits are separated by more than 1e-4 of the router's
sum |R x| (ambiguous tokens are counted and reported).
"""
import numpy as np

AMBIGUITY = 1e-4


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


def check_moe(out_gpu, idx_gpu, w_gpu, ref, what="moe"):
    """ref: dict from oracle.moe_ffn.  Returns the number of ambiguous tokens."""
    out_gpu = np.asarray(out_gpu).reshape(ref["out"].shape)
    idx_gpu = np.asarray(idx_gpu).reshape(ref["idx"].shape)
    amb = ref["gap"] <= AMBIGUITY
    for t in range(idx_gpu.shape[0]):
        if amb[t]:
            continue
        if not np.array_equal(idx_gpu[t], ref["idx"][t]):
            raise ParityError(f"{what}: token {t} routed to {idx_gpu[t].tolist()}, "
                              f"oracle {ref['idx'][t].tolist()}")
    if w_gpu is not None:
        w_gpu = np.asarray(w_gpu).reshape(ref["w"].shape)
        check_close(w_gpu[~amb], ref["w"][~amb], 1e-5 * np.abs(ref["w"][~amb]) + 1e-6,
                    f"{what} routing weights")
    check_close(out_gpu[~amb], ref["out"][~amb], ref["tol"][~amb], f"{what} residual")
    return int(np.sum(amb))
