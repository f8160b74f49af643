"""Host-side arithmetic of the benchmark line (CPU only): bytes per quantised
position for each code width, the algorithmic bytes of one decode call (the
sum of its parts, checked at the Llama-shaped 32K layer), the period mean,
and the rule that the recorded DRAM traffic is used only for the kernel
source it was measured on."""
import hashlib
import json
import os

import bench


def test_quantised_row_bytes_per_width():
    # K and V: 128 codes of B bits each, plus four (scale, zero) FP16 pairs
    assert bench.q_row_bytes(4, 4) == 2 * (64 + 16) == 160
    assert bench.q_row_bytes(8, 8) == 2 * (128 + 16) == 288
    assert bench.q_row_bytes(4, 8) == bench.q_row_bytes(8, 4) == (64 + 16) + (128 + 16) == 224


def test_algorithmic_bytes_of_the_32k_layer():
    P = 32768 - 128
    k = -(-P * 50_000 // 1_000_000)        # ceil(rho P) vertical lines
    n_q, n_tail = P - k, 128
    want = 8 * (n_q * 160 + (k + n_tail) * 2 * 128 * 2) + 2 * 32 * 128 * 2
    assert k == 1632 and n_q == 31008
    assert bench.algorithmic_bytes(n_q, k, n_tail) == want == 46_915_584   # 46.9 MB with a 128-row tail
    assert bench.algorithmic_bytes(n_q, k, n_tail, bench.q_row_bytes(8, 8)) == want + 8 * n_q * (288 - 160)


def test_period_mean_lies_between_its_first_and_last_call():
    P0 = bench.L0 - bench.WINDOW
    k0 = -(-P0 * bench.RHO_PPM // 1_000_000)
    first = bench.algorithmic_bytes(P0 - k0, k0, bench.WINDOW + 1)
    last_tail = bench.algorithmic_bytes(P0 - k0, k0, bench.WINDOW + bench.PERIOD - 1)
    mean = bench.period_bytes_per_decode()
    assert first < mean < max(last_tail, bench.algorithmic_bytes(bench.CTX - bench.WINDOW - k0, k0, bench.WINDOW))
    assert bench.period_bytes_per_decode(288) > mean


def test_traffic_record_is_used_only_for_its_source(tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "decode_attention_llama32k_traffic.json")))
    src = open(os.path.join(bench.ROOT, "hybrid_precision_quantized_gb300", "csrc", "hyq_decode.cu"), "rb").read()
    if rec["kernel_source_sha256"] == hashlib.sha256(src).hexdigest():
        assert bench.decode_traffic() == float(rec["dram_bytes_per_launch"])
    else:                                   # taken on another source: reported as unknown
        assert bench.decode_traffic() is None
    # a copy of the tree whose kernel source differs reports no traffic
    (tmp_path / "profiles").mkdir()
    (tmp_path / "hybrid_precision_quantized_gb300" / "csrc").mkdir(parents=True)
    (tmp_path / "profiles" / "decode_attention_llama32k_traffic.json").write_text(json.dumps(rec))
    (tmp_path / "hybrid_precision_quantized_gb300" / "csrc" / "hyq_decode.cu").write_bytes(src + b"\n// changed\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.decode_traffic() is None
