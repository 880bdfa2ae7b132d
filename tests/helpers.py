"""Shared test helpers: tolerances, comparison against the oracle, input prep."""
import numpy as np
import torch

import oracle
from paged_kv_decode_21_gb300 import workloads

# fp16 output, fp32 accumulation: element-wise bound and mean bound against
# the fp64 oracle (the library's stated parity contract).
MAX_ABS_TOL = 4e-3
MEAN_ABS_TOL = 5e-4


def oracle_out(inp: workloads.DecodeInputs, rows=None, threads=None):
    return oracle.attention(inp.q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), inp.block_tables.cpu(),
                            inp.context_lens.cpu(), inp.scale, rows=rows, threads=threads)


def assert_close(got_fp16: torch.Tensor, ref: np.ndarray, what=""):
    got = got_fp16.detach().cpu().to(torch.float64).numpy()
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    assert mx <= MAX_ABS_TOL and mean <= MEAN_ABS_TOL, f"{what}: max|err|={mx:.3e} mean|err|={mean:.3e}"
    return mx, mean


def sample_rows(num_seqs, num_q_heads, n, seed=0):
    rng = np.random.default_rng(seed)
    total = num_seqs * num_q_heads
    n = min(n, total)
    rows = rng.choice(total, size=n, replace=False).astype(np.int32)
    # always include the first and last rows
    rows[0] = 0
    rows[-1] = total - 1
    return np.unique(rows)


def e4m3_magnitudes(codes8: torch.Tensor) -> torch.Tensor:
    """E4M3 codes with the sign bit cleared: attention over them gives
    sum_t w_t |v_t|, since the weights w_t do not depend on V."""
    return codes8 & 0x7F


def assert_close_weighted(got_fp16: torch.Tensor, ref: np.ndarray, absref: np.ndarray, vmax: float,
                          max_len: int, what=""):
    """The tolerance above, plus an element bound from the arithmetic of the
    tensor-core paths: each weight p is rounded to fp16 before P.V (relative
    error 2^-11, or 2^-25 absolute where p is an fp16 subnormal) and the
    output once to fp16 (2^-11 relative); fp32 rounding elsewhere is far
    smaller.  With absref = sum_t w_t |v_t| (the oracle over |V|), vmax the
    largest |v| and max_len the longest context, every element must satisfy
    |err| <= 2^-9 absref + 2^-10 |ref| + 2^-24 max_len vmax (4x the
    first-order terms, 2x the last), so a wrong weight or term shows even
    where the outputs are far below the absolute tolerance."""
    mx, mean = assert_close(got_fp16, ref, what)
    got = got_fp16.detach().cpu().to(torch.float64).numpy()
    err = np.abs(got - ref)
    bound = 2.0 ** -9 * absref + 2.0 ** -10 * np.abs(ref) + 2.0 ** -24 * max_len * vmax
    worst = float((err / bound).max(initial=0.0))
    assert worst <= 1.0, f"{what}: error {worst:.2f}x the element bound (max|err|={mx:.3e})"
    return mx, mean, worst
