"""The bench's printed line, built on the CPU from figures shaped like a full
run's: it carries the contract's keys and stays short enough for a log tail
that keeps about 3,000 characters."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_the_default_line_fits_the_budget():
    sys.path.insert(0, ROOT)
    import bench
    sys.argv = ["bench.py"]
    args = bench.parse()
    names = ([f"global_{c}" for c in args.contexts] + [f"window_{bench.WINDOW_RESIDENCY}"]
             + [f"folded_{c}" for c in args.folded_contexts]
             + [f"verify_{args.verify_context}x{t}" for t in args.verify_tokens]
             + [f"tree_{args.verify_context}x{t}" for t in args.tree_tokens] + ["ragged16"])
    big = dict(us_per_call=1234.56, GBps_per_call=12345.6, frac_of_8TBs=1.2345,
               frac_of_measured=1.2345, splits=1024, partial_us=1234.56, us_stream=1234.56,
               us_isolated=1234.56)
    detail = {n: dict(big) for n in names}
    sweep = {n: {"us": {p: 12345.67 for p in args.sweep}, "best_splits": 256}
             for n in names if n.startswith("global")}
    prefill = {f"prefill_{p.replace(':', '_')}": {"tflops": 1234.5} for p in args.prefill}
    roofline = {"bound": "hbm", "kernel": "pskv_partial_kernel<MmaConsumer<512, 8>>",
                "achieved": 12345.6, "peak": 6784.5, "unit": "GB/s", "frac": 1.2345,
                "peak_source": "measured hbm_gbs", "algorithmic_bytes_per_launch": 605374464.0,
                "traffic": 611411951}
    e2e = {"value": 12345.6, "unit": "GB/s", "ms_per_step": 1.23456,
           "h2d_bytes_per_step": 1234567, "d2h_bytes_per_step": 1234567,
           "how": "eager C-ABI calls; one packed copy in, one out per step"}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 60,
              "reasons": ["sw_power_cap"],
              "window": "every 100 ms: 0.4 s before the timed steps, them, 0.2 s after"}
    line = bench.make_line(args, 8, 12345.67, 1.23456, 123456, roofline, e2e, clocks,
                           {"graph": 1.23456, "eager": 1.23456, "prep": 1.23456}, detail,
                           sweep, prefill)
    line["cpu_baseline"] = {"value": 12.345, "unit": "GB/s", "cores": 128, "kind": "oracle",
                            "sample": "123 passes of the step's 5 calls (10602/40002/81653/"
                                      "163336/1088 keys), fp64 direct softmax, 12.3 s"}
    text = json.dumps(line, separators=(",", ":"), ensure_ascii=False)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "gpu_launches", "roofline", "e2e", "clocks", "cpu_baseline"):
        assert key in line
    print("line length", len(text))
    assert len(text) <= bench.LINE_BUDGET, len(text)
