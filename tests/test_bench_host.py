"""Host-side helpers of bench.py: the clock summary and the step-time summary."""
import bench


def test_clock_summary_decodes_reason_bits():
    lines = ["0, 2070, 2070, 0x0000000000000000",
             "0, 1965, 2070, 0x0000000000000004",          # sw power cap
             "0, 2070, 2070, 0x0000000000000048",          # hw slowdown + hw thermal
             "0, [N/A], 2070, 0x0000000000000020",         # unreadable clock: skipped
             "garbage"]
    s = bench.ClockSampler.summarize(lines)
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]


def test_clock_summary_without_samples():
    assert bench.ClockSampler.summarize([])["reasons"] == ["no samples"]


def test_step_time_summary_counts_stalls():
    t = [0.1] * 50 + [1000.1]
    s = bench.step_time_summary(t)
    assert s["median_ms"] == 0.1 and s["stalled_steps"] == 1 and abs(s["stalled_ms"] - 1000.0) < 1e-6
    assert bench.step_time_summary([0.1] * 10)["stalled_steps"] == 0


def test_code_hash_ignores_comments_and_layout():
    """A committed ncu traffic figure stays valid across comment edits, not
    across code edits: the hash covers the code with comments and blank space
    removed, string and character literals kept."""
    a = 'int f(int x) {\n    // one\n    return x + 1;  /* two */\n}\nconst char* s = "// kept";\n'
    b = 'int f(int x) { return x + 1; }\n/* another comment */ const char* s = "// kept";'
    c = 'int f(int x) { return x + 2; }\nconst char* s = "// kept";'
    d = 'int f(int x) { return x + 1; }\nconst char* s = "// changed";'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert bench._code_only(a) != bench._code_only(d)
    assert bench._code_only("char c = '/'; // x") == "char c = '/';"

