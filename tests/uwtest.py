"""Helpers shared by the GPU tests: device buffers, the matmul tolerance (1e-4 of sum |w x| plus 1e-6; 2^-7
relative added for bf16 output), the rows a full-size parity test checks, and a cache of the oracle's results."""
import numpy as np

import lossless_bf16_weight_exponent_gb300 as uw
import oracle


def torch():
    import torch as t
    return t


def to_dev_u16(a: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def dev_bytes(n: int):
    t = torch()
    return t.empty(max(int(n), 16), dtype=t.uint8, device="cuda")


def tol_ok(y, yref, absum, bf16_out=False):
    """|y - yref| <= 1e-4 * sum_k |w x| + 1e-6  (fp32 out);  + 2^-7 |yref| after bf16 rounding."""
    bound = 1e-4 * absum + 1e-6
    if bf16_out:
        bound = bound + 2.0 ** -7 * np.abs(yref)
    err = np.abs(y.astype(np.float64) - yref)
    return bool((err <= bound).all()), float((err / np.maximum(bound, 1e-300)).max())


def run_matmul(m, x_np, plan_or_strategy, out_dtype=uw.OUT_F32, stream=None):
    """Run one uw_matmul (plan tuple or strategy int) and return Y as numpy float64."""
    t = torch()
    B = x_np.shape[0]
    x = to_dev_u16(x_np)
    if isinstance(plan_or_strategy, tuple):
        plan = uw.Plan(*plan_or_strategy)
        nbytes = m.plan_workspace_size(B, plan)
    else:
        plan = None
        nbytes = m.workspace_size(B, plan_or_strategy)
    ws = dev_bytes(nbytes)
    if out_dtype == uw.OUT_F32:
        y = t.full((B, m.N), float("nan"), dtype=t.float32, device="cuda")
    else:
        y = t.full((B, m.N), float("nan"), dtype=t.bfloat16, device="cuda")
    if plan is not None:
        m.matmul_plan(x, B, y, plan, out_dtype, ws, nbytes)
    else:
        m.matmul(x, B, y, out_dtype, plan_or_strategy, ws, nbytes)
    t.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64)


def strategies_for(m):
    out = [uw.STRAT_FULL_DECODE, uw.STRAT_EXP_ONLY]
    if m.info["has_huffman_stream"]:
        out.append(uw.STRAT_PALETTE_TRANSCODE)
    if m.info["has_palette_form"]:
        out.append(uw.STRAT_DIRECT_PALETTE)
    return out


def check_rows(N, B, seed=0):
    """Rows a full-size parity test compares: every row when B <= 4 (the oracle's fp64 GEMV of the 8B gate_proj
    takes about a second per batch row); otherwise one random row from each of 1024 equal bins of [0, N) plus the
    first and last two rows, so every CTA's and every 128-row unit's row range is checked."""
    if B <= 4 or N <= 2048:
        return None
    rng = np.random.default_rng(seed)
    edges = np.linspace(0, N, 1025).astype(np.int64)
    picks = [int(rng.integers(lo, hi)) for lo, hi in zip(edges[:-1], edges[1:]) if hi > lo]
    return np.unique(np.array([0, 1, N - 2, N - 1] + picks, dtype=np.int64))


_REF = {}


def oracle_ref(key, w, x, rows=None):
    """The oracle's (Y, sum |w x|) for these rows (None: all), cached by key so tests sharing a full-size
    workload pay for its fp64 contraction once."""
    k = (key, x.shape[0], None if rows is None else rows.tobytes())
    if k not in _REF:
        _REF[k] = oracle.matmul(w, x, rows)
    return _REF[k]


def pick(y, rows):
    """Y restricted to the checked rows (all rows when rows is None)."""
    return y if rows is None else y[:, rows]
