"""Host-side checks of bench.py: it parses, and its reference arm (the fp64 oracle on the host
cores) prints one JSON line carrying the keys of the benchmark line."""
import ast
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_parses():
    with open(os.path.join(ROOT, "bench.py")) as f:
        ast.parse(f.read())


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_zipf_workload_is_skewed():
    """The skewed-popularity workload (tiny layer shape, T=8192, Zipf(1.1) bias channel):
    the bias channel survives margin redraws and expert popularity falls with the index."""
    import numpy as np

    import oracle
    from mixture_experts_layer_09_gb300 import inputs as gen
    import workloads as wk

    inp = wk.layer("tiny_zipf_t8192")
    assert np.all(inp.x[:, 0] == gen.ONE_BF16)
    ids, _ = oracle.router_topk(oracle.router_logits(inp.x, inp.W_r), inp.wl.k)
    share = np.bincount(ids.ravel(), minlength=inp.wl.E) / ids.size
    assert share[0] > 0.3 and share[0] > 4 * share[-1]
    assert np.all(np.diff(share[:4]) < 0)  # the head of the distribution is strictly ordered


def test_algorithmic_bytes_match_the_uploaded_arrays():
    """The roofline's bytes per expert equal what one expert's three matrices occupy in the
    layout the kernels stream (codes plus a 2-byte scale per 32 columns), for both formats;
    the MXFP4 upload turns each exponent byte into a 2-byte scale."""
    import numpy as np

    sys.path.insert(0, ROOT)
    import bench
    from mixture_experts_layer_09_gb300 import inputs as gen
    for H, I in ((256, 128), (2048, 768), (6144, 2048)):
        for fmt in ("int4", "mxfp4"):
            ex = gen.draw_experts(3, 1, H, I, fmt)
            q_bytes = sum(m.q.nbytes for m in (ex.gate, ex.up, ex.down))
            s_elems = sum(m.s.size for m in (ex.gate, ex.up, ex.down))
            assert bench.BYTES_PER_EXPERT(H, I) == q_bytes + 2 * s_elems, (H, I, fmt)
    # the per-expert figures the measurement plan quotes
    assert bench.BYTES_PER_EXPERT(2048, 768) == 2_654_208
    assert bench.BYTES_PER_EXPERT(6144, 2048) == 21_233_664
    assert bench.BYTES_PER_EXPERT(2048, 1408) == 4_866_048
    assert np.isclose(bench.BYTES_PER_EXPERT(2048, 5632), 19_464_192)
