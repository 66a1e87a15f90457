"""Host-side helpers of bench.py that need no GPU."""
import os

import bench


def _write(tmp_path, name, text):
    p = os.path.join(tmp_path, name)
    with open(p, "w") as f:
        f.write(text)
    return p


def test_code_hash_ignores_comments_and_blank_lines_only(tmp_path):
    base = _write(tmp_path, "a.cu", 'int a = 1;  // one\n/* two */\nconst char* s = "// kept";\n')
    comments = _write(tmp_path, "b.cu", '// header\nint a = 1;  // changed\n\n/* two\n lines */\nconst char* s = "// kept";\n')
    code = _write(tmp_path, "c.cu", 'int a = 2;  // one\n/* two */\nconst char* s = "// kept";\n')
    string = _write(tmp_path, "d.cu", 'int a = 1;  // one\n/* two */\nconst char* s = "// other";\n')
    assert bench.code_hash(base) == bench.code_hash(comments)
    assert bench.code_hash(base) != bench.code_hash(code)
    assert bench.code_hash(base) != bench.code_hash(string)  # text inside a string literal is code


def test_recorded_traffic_entries_are_well_formed():
    path = os.path.join(bench.ROOT, "profiles", "traffic.txt")
    for ln in open(path):
        if ln.startswith("#") or not ln.strip():
            continue
        workload, src, h, nbytes = ln.split()
        assert workload in bench.WORKLOADS or workload in bench.GATHER_WORKLOADS
        assert os.path.exists(os.path.join(bench.ROOT, "block_quantized_moe_gb300", src))
        assert len(h) == 12 and int(h, 16) >= 0 and int(nbytes) > 0
    assert bench.recorded_traffic("no-such-workload") is None


def test_vs_baseline_only_for_workloads_the_pages_time():
    assert bench.vs_pages("decode-h4096-i1024-e64-t8-a8", 118.0) is None  # no page number
    assert bench.vs_pages(bench.DEFAULT_WORKLOAD, 3000.0) is None
    assert bench.vs_pages("decode-h2048-i768-e8-t1-a2", 60.589) == 1.0
    assert bench.vs_pages("gather-k7168-t1024", 5.57) == 0.5
    for name in bench.PAGES_US:
        assert name in bench.WORKLOADS or name in bench.GATHER_WORKLOADS


def test_cpu_baseline_oracle_call_equals_the_numpy_oracle():
    # the bench's CPU-baseline call (C++ oracle over a bank compacted to the used experts)
    # computes the numpy oracle's forward, in every format and with no active route
    import numpy as np

    import synth
    from oracle import moe as M
    T, H, I, E, k, seed = 4, 256, 128, 6, 3, 5
    x = synth.activations_bf16(T, H, seed, "cpu").float().numpy()
    ids = synth.routes(T, k, E, seed, active_per_token=[3, 2, 0, 3], device="cpu").numpy()
    w = synth.routing_weights(T, k, seed, "cpu").numpy()
    used = sorted(set(int(e) for e in ids.reshape(-1) if e >= 0))
    for fmt in ("fp8", "nvfp4", "mxfp8"):
        bg = M.LazyBank(lambda e: synth.expert_weight_fp32(2 * I, H, seed, e, "gateup", "cpu").numpy(), 2 * I, fmt)
        bd = M.LazyBank(lambda e: synth.expert_weight_fp32(H, I, seed, e, "down", "cpu").numpy(), H, fmt)
        got = bench._cpp_oracle_call(x, ids, w, used, fmt, H, I, seed=seed)(4)
        ref = M.moe_forward(x, ids, w, bg, bd, fmt=fmt)["out"]
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-14 * np.abs(ref).max())
        none = np.full_like(ids, -1)
        assert not bench._cpp_oracle_call(x, none, w, [], fmt, H, I, seed=seed)(2).any()


def test_cpu_baseline_uses_the_cpp_oracle_and_falls_back_to_numpy(monkeypatch):
    res = bench.cpu_baseline("decode-h2048-i768-e8-t1-a2", budget_s=1.0, min_s=0.2)
    assert res["kind"] == "oracle" and res["value"] > 0 and "C++ oracle" in res["sample"]
    from oracle import cpu as C

    def unavailable():
        raise RuntimeError("no compiler")
    monkeypatch.setattr(C, "lib", unavailable)
    res = bench.cpu_baseline("decode-h2048-i768-e8-t1-a2", budget_s=1.0, min_s=0.2)
    assert res["cores"] == 1 and "numpy" in res["sample"] and "no compiler" in res["sample"]
