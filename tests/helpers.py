"""Shared test helpers: tolerances, comparisons, host copies, and a runner
that checks every token of a large call against the oracle on all host
cores.  No finalize arithmetic lives here."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle

# FP32 residual: |gpu - oracle| <= max(REL * |oracle|, ABS) per element
RES_REL = 1e-6
RES_ABS = 1e-6
# bf16 output: at most this many units in the last place apart
OUT_ULP = 1


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def bf16_ordered(b: np.ndarray) -> np.ndarray:
    """Maps bf16 bit patterns to integers whose order is the value order;
    +0 and -0 both map to 0."""
    b = b.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_is_nan(b: np.ndarray) -> np.ndarray:
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    d = np.abs(bf16_ordered(a) - bf16_ordered(b)).astype(np.float64)
    na, nb = bf16_is_nan(a), bf16_is_nan(b)
    d[na & nb] = 0
    d[na ^ nb] = np.inf
    return d


def assert_residual_close(got: np.ndarray, want: np.ndarray, what="residual_out"):
    got = np.asarray(got, dtype=np.float32)
    want = np.asarray(want, dtype=np.float32)
    if got.shape != want.shape:
        raise AssertionError(f"{what}: shape {got.shape} != {want.shape}")
    if np.array_equal(got.view(np.uint32), want.view(np.uint32)):
        return                                   # bit-equal: within any tolerance
    both_nan = np.isnan(got) & np.isnan(want)
    with np.errstate(invalid="ignore"):
        err = np.abs(got.astype(np.float64) - want.astype(np.float64))
        tol = np.maximum(RES_REL * np.abs(want.astype(np.float64)), RES_ABS)
        bad = ~both_nan & ~(err <= tol) & ~(got == want)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; first at {tuple(i)}: "
                             f"got {got[tuple(i)]!r} want {want[tuple(i)]!r}")


def assert_out_close(got_bits: np.ndarray, want_bits: np.ndarray, what="out", ulp=OUT_ULP):
    if got_bits.shape != want_bits.shape:
        raise AssertionError(f"{what}: shape {got_bits.shape} != {want_bits.shape}")
    d = bf16_ulp_distance(got_bits, want_bits)
    if not np.all(d <= ulp):
        i = np.argwhere(~(d <= ulp))[0]
        raise AssertionError(f"{what}: {(~(d <= ulp)).sum()} elements beyond {ulp} ulp; first at {tuple(i)}: "
                             f"got 0x{int(got_bits[tuple(i)]):04x} want 0x{int(want_bits[tuple(i)]):04x}")


def oracle_on(inputs: dict, tokens=None, residual=None):
    """Runs the oracle on host copies of the inputs (optionally on a subset
    of tokens).  Returns (residual_out, out_bits, bad_slots)."""
    res = f32(inputs["residual"] if residual is None else residual)
    return oracle.finalize_residual_rmsnorm(
        bf16_bits(inputs["expert_out"]), inputs["permuted_row_of"].cpu().numpy(),
        f32(inputs["topk_weights"]), res, bf16_bits(inputs["gamma"]), inputs["eps"], tokens=tokens)


def oracle_finalize_only(inputs: dict, tokens=None):
    """The oracle's plain finalize on host copies: (out_bits, bad_slots)."""
    return oracle.finalize_only(bf16_bits(inputs["expert_out"]), inputs["permuted_row_of"].cpu().numpy(),
                                f32(inputs["topk_weights"]), tokens=tokens)


def oracle_expert_norm(inputs: dict, tokens=None):
    """The oracle's per-expert RMSNorm finalize on host copies:
    (out_bits, y float64, s float64, bad_slots), where y is the exact value
    before rounding and s the same sum over |w|, |E| and |gamma| (the scale
    of the FP32 rounding error of any evaluation order)."""
    E = bf16_bits(inputs["expert_out"])
    idx = inputs["permuted_row_of"].cpu().numpy()
    w = f32(inputs["topk_weights"])
    g = bf16_bits(inputs["gamma"])
    out, bad = oracle.finalize_expert_rmsnorm(E, idx, w, g, inputs["eps"], tokens=tokens)
    y, _ = oracle.expert_rmsnorm_f64(E, idx, w, g, inputs["eps"], tokens=tokens)
    s, _ = oracle.expert_rmsnorm_f64(E & np.uint16(0x7FFF), idx, np.abs(w), g & np.uint16(0x7FFF),
                                     inputs["eps"], tokens=tokens)
    return out, y, s, bad


# ---- every token of a large call, on all host cores ------------------------------

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_inputs(inputs: dict) -> dict:
    """Host copies of a call's inputs, made once: bf16 as uint16 bits."""
    return {"E": bf16_bits(inputs["expert_out"]), "idx": inputs["permuted_row_of"].cpu().numpy(),
            "w": f32(inputs["topk_weights"]), "res": f32(inputs["residual"]), "gamma": bf16_bits(inputs["gamma"]),
            "eps": inputs["eps"]}


def over_all_tokens(T: int, check, chunk: int = 256, threads=None) -> int:
    """Calls check(tokens) for consecutive chunks of [0, T) on a pool of host
    threads (the oracle's C calls and NumPy's large-array operations release
    the GIL) and re-raises the first failure.  Returns the tokens covered."""
    chunks = [np.arange(a, min(a + chunk, T), dtype=np.int64) for a in range(0, T, chunk)]
    with ThreadPoolExecutor(max_workers=threads or host_cores()) as ex:
        for _ in ex.map(check, chunks):
            pass
    return int(sum(c.size for c in chunks))


def check_every_token(h: dict, got_res: np.ndarray, got_out: np.ndarray, chunk: int = 256) -> int:
    """The fused path's outputs (residual_out f32 [T, H], out bf16 bits
    [T, H]) against the oracle, token by token over all T tokens."""
    T = h["idx"].shape[0]

    def check(tk):
        want_res, want_out, bad = oracle.finalize_residual_rmsnorm(h["E"], h["idx"], h["w"], h["res"], h["gamma"],
                                                                   h["eps"], tokens=tk)
        assert bad == 0
        assert_residual_close(got_res[tk[0]:tk[-1] + 1], want_res, what=f"residual_out tokens {tk[0]}..")
        assert_out_close(got_out[tk[0]:tk[-1] + 1], want_out, what=f"out tokens {tk[0]}..")
    return over_all_tokens(T, check, chunk)


def check_every_token_finalize_only(h: dict, got_out: np.ndarray, chunk: int = 256) -> int:
    """The plain finalize's bf16 output against the oracle's, bit for bit,
    over all T tokens."""
    T = h["idx"].shape[0]

    def check(tk):
        want, bad = oracle.finalize_only(h["E"], h["idx"], h["w"], tokens=tk)
        assert bad == 0
        got = got_out[tk[0]:tk[-1] + 1]
        if not np.array_equal(got, want):
            i = np.argwhere(got != want)[0]
            raise AssertionError(f"finalize out differs at token {tk[0] + i[0]}, column {i[1]}")
    return over_all_tokens(T, check, chunk)
