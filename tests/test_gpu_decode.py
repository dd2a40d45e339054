"""Decode attention on the GPU against the CPU oracle.

* The five workloads at full size, in the launch configuration the benchmark
  uses (heuristic split), every sequence and every head compared with the
  oracle; all 16 ragged long-context trials on their longest and shortest
  sequences.
* Random small shapes spanning several tiles and a ragged tail, every
  supported head dimension and a range of group sizes, with forced split
  counts 1, 2, 3, 7 and more CTAs than tokens.
* Edge cases: empty and one-token sequences, lengths clamped on the device,
  NaN-filled cache padding (any read past a sequence's end poisons the
  output), guard bands around the outputs and the workspace, and bitwise
  determinism across runs.
Tolerances: bf16 output within 1e-2; an element above it must lie within half
a bf16 step at its magnitude plus the bound on the bf16 weights' rounding
(gpu_helpers.assert_close), and the count of such elements is recorded; fp32
output within 1e-4. The natural-log normaliser lse within 1e-4 in
fp32 mode; in bf16 mode the normaliser sums the bf16-rounded weights (the ones
multiplied into V, so that the output stays an exact convex combination of V
rows), which carry up to 2^-9 relative rounding each, so lse is held to 2^-8.
"""
import numpy as np
import pytest

import workloads
from gpu_helpers import assert_close, cuda_or_skip, oracle_step, run_step, spread_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def _check(inp, r, out_dtype, rows=None, what=""):
    ref, ref_lse = oracle_step(inp, rows)
    got = r.out if rows is None else r.out[np.asarray(rows)]
    lse = r.lse if rows is None else r.lse[np.asarray(rows)]
    err = assert_close(got, ref, out_dtype, what, spread=spread_step(inp, rows))
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), what
    lse_tol = 1e-4 if out_dtype == "f32" else 2.0 ** -8
    assert np.max(np.abs(lse[fin] - ref_lse[fin]), initial=0.0) < lse_tol, what
    assert np.all(lse[~fin] == -np.inf), what
    assert r.guards_ok, f"{what}: output guard band overwritten"
    assert r.ws_guards_ok, f"{what}: workspace guard band overwritten"
    return err


# ---------------------------------------------------------------------------
# Full-size workloads
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def full_inputs():
    cache = {}

    def get(name):
        if name not in cache:
            cache.clear()  # keep one full-size workload in host memory at a time
            cache[name] = workloads.step_inputs(workloads.get(name))
        return cache[name]
    return get


@pytest.mark.parametrize("name", ["tiny", "palm", "mha", "gqa", "long"])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_workload_full_size(dev, full_inputs, name, out_dtype):
    inp = full_inputs(name)
    r = run_step(inp, dev, out_dtype)
    assert r.status == 0
    _check(inp, r, out_dtype, None, f"{name}/{out_dtype}/n_split={r.n_split}")


@pytest.mark.parametrize("trial", range(16))
def test_long_ragged_trial(dev, trial):
    w = workloads.long_trial(trial)
    inp = workloads.step_inputs(w)
    r = run_step(inp, dev, "bf16", max_seq_len=w.S_max)
    rows = [int(np.argmax(inp.seq_lens)), int(np.argmin(inp.seq_lens))]
    _check(inp, r, "bf16", rows, f"long_trial{trial}")


@pytest.mark.parametrize("n_split", [1, 7, 1000])
def test_palm_forced_splits(dev, full_inputs, n_split):
    inp = full_inputs("palm")
    r = run_step(inp, dev, "bf16", n_split=n_split)
    _check(inp, r, "bf16", [0, 40, 63], f"palm n_split={n_split}")


# ---------------------------------------------------------------------------
# Small shapes: brute force against the oracle on every element
# ---------------------------------------------------------------------------

SMALL = [  # (seed, B, Hq, Hkv, D, S_max, lens)
    (1, 3, 8, 1, 128, 300, [300, 1, 157]),
    (2, 4, 4, 4, 64, 200, [200, 0, 65, 64]),
    (3, 2, 6, 2, 128, 97, [97, 33]),
    (4, 2, 16, 1, 256, 130, [130, 17]),
    (5, 5, 40, 8, 128, 90, [90, 0, 1, 45, 89]),
    (6, 2, 17, 1, 64, 70, [70, 3]),
    (7, 2, 48, 1, 256, 300, [300, 129]),
    (8, 3, 64, 1, 128, 100, [99, 100, 2]),
    (9, 2, 33, 1, 64, 50, [50, 31]),
    (10, 2, 96, 2, 256, 80, [80, 41]),
    (11, 6, 32, 8, 128, 64, [64, 0, 0, 1, 63, 32]),
    (12, 1, 1, 1, 64, 513, [513]),
]


@pytest.mark.parametrize("case", SMALL, ids=[f"s{c[0]}_G{c[2] // c[3]}_D{c[4]}" for c in SMALL])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_small_shapes(dev, case, out_dtype):
    seed, B, Hq, Hkv, D, S, lens = case
    inp = workloads.random_small(seed, B, Hq, Hkv, D, S, lens)
    for n_split in (0, 1, 2, 3, 7, 10000):
        r = run_step(inp, dev, out_dtype, n_split=n_split)
        assert r.status == 0
        _check(inp, r, out_dtype, None, f"seed{seed}/{out_dtype}/n_split={n_split}")


def test_peaked_small(dev):
    inp = workloads.step_inputs(workloads.Workload("pk", 4, 32, 8, 128, 500, 100, 500, 77,
                                                   peaked_frac=0.05))
    for out_dtype in ("bf16", "f32"):
        r = run_step(inp, dev, out_dtype)
        _check(inp, r, out_dtype, None, f"peaked/{out_dtype}")


# ---------------------------------------------------------------------------
# Edge cases
# ---------------------------------------------------------------------------

def test_all_empty(dev):
    inp = workloads.random_small(20, 3, 8, 2, 64, 16, [0, 0, 0])
    for n_split in (0, 1, 5):
        r = run_step(inp, dev, "bf16", n_split=n_split, max_seq_len=16)
        assert np.all(r.out == 0.0) and np.all(r.lse == -np.inf)
        assert r.guards_ok and r.ws_guards_ok


def test_lengths_clamped_on_device(dev):
    import kv_cache_decode_gb300 as kvd
    inp = workloads.random_small(21, 4, 8, 1, 128, 64, [64, 10, 30, 1])
    bad = np.array([500, -7, 30, 1], np.int32)      # 500 > max_seq_len, -7 < 0
    r = run_step(inp, dev, "f32", max_seq_len=40, seq_lens_override=bad)
    assert r.status & kvd.STATUS_SEQ_LEN_CLAMPED
    clamped = np.clip(bad, 0, 40)
    ref, _ = oracle_step(inp, lens=clamped)
    assert_close(r.out, ref, "f32", "clamped")


def test_deterministic(dev, full_inputs):
    inp = full_inputs("palm")
    a = run_step(inp, dev, "bf16")
    b = run_step(inp, dev, "bf16")
    assert np.array_equal(a.out, b.out) and np.array_equal(a.lse, b.lse)
