"""Host-side logic of bench.py (no GPU): clock-sample parsing, repetition
count of the timed region, and the config object both arms print."""
import importlib.util
import os

from decode_attention_paged_pa_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


ROW = "GPU-{u}, {sm}, 2070, 900.5, 0x0000000000000000, {hw}, Not Active, Not Active, {cap}"


def test_clock_rows_of_our_gpu_only():
    b = _bench()
    ours = "11111111-2222-3333-4444-555555555555"
    lines = [ROW.format(u=ours, sm=2070, hw="Not Active", cap="Not Active"),
             ROW.format(u="aaaaaaaa-2222-3333-4444-555555555555", sm=900, hw="Active", cap="Active"),
             ROW.format(u=ours, sm=2055, hw="Not Active", cap="Active"),
             ROW.format(u=ours, sm=2070, hw="Not Active", cap="Not Active")]
    got = b.summarize_clocks(lines, ours)
    assert got["samples"] == 3
    assert got["sm_mhz"] == 2070 and got["sm_max_mhz"] == 2070
    assert got["reasons"] == ["sw_power_cap"]          # the other GPU's hw_slowdown is not ours


def test_clock_rows_single_gpu_without_uuid_match():
    b = _bench()
    lines = [ROW.format(u="abcdef01-2222-3333-4444-555555555555", sm=s, hw="Not Active", cap="Not Active")
             for s in (1900, 2000, 2070)]
    got = b.summarize_clocks(lines, "")
    assert got["samples"] == 3 and got["sm_mhz"] == 2000 and got["reasons"] == []
    # two GPUs and no way to tell ours: nothing rather than a wrong GPU's clocks
    two = lines + [ROW.format(u="ffffffff-2222-3333-4444-555555555555", sm=1000, hw="Active", cap="Active")]
    assert b.summarize_clocks(two, "")["samples"] == 0
    assert b.summarize_clocks(["garbage", ""], "")["samples"] == 0


def test_repetitions_cover_the_minimum_time():
    b = _bench()
    assert b.repetitions_needed(12.0, 1.0) == 84          # 84 x 12 ms >= 1 s
    assert b.repetitions_needed(2000.0, 1.0) == 1
    assert b.repetitions_needed(0.01, 1.0, cap=50) == 50
    assert b.repetitions_needed(0.0, 1.0) == 1


def test_both_arms_print_the_same_config():
    b = _bench()
    w = workloads.WORKLOADS[b.HEADLINE]
    c = b.config_of(w, 1, "auto")
    assert c["workload"] == "d256_fp16" and c["head_size"] == 256
    assert c == b.config_of(w, 1, "auto", b.expected_lens(w))
    # the headline is the largest of the five configurations by bytes moved
    sizes = {n: workloads.algorithmic_bytes(workloads.WORKLOADS[n], b.expected_lens(workloads.WORKLOADS[n]))
             for n in b.BASE_CONFIGS}
    assert max(sizes, key=sizes.get) == b.HEADLINE
    # pools smaller than L2 are flushed between timed calls, larger ones are not
    assert "flushed" in b.config_of(workloads.WORKLOADS["tiny_fp16"], 1, "auto")["l2"]
    assert "no flush" in c["l2"]
