"""The benchmark's link to the committed ncu summaries (CPU only).

`bench.py` reports a kernel's DRAM traffic from `profiles/` only while the summary's
source digest matches the code the kernel is built from. The digest covers the code with its
comments and blank lines removed: a comment edit keeps a capture valid, a code edit does not.
"""
import os

import bench


def test_code_only_drops_comments_and_blank_lines_but_keeps_literals():
    src = ('int a = 1;  // note\n'
           '\n'
           '/* block\n   comment */ const char* s = "a // b /* c */";\n'
           "char q = '\"'; char r = '\\'';  /* tail */\n")
    assert bench._code_only(src) == ('int a = 1;\n'
                                     ' const char* s = "a // b /* c */";\n'
                                     "char q = '\"'; char r = '\\'';")


def test_digest_follows_code_not_comments(tmp_path, monkeypatch):
    pkg = tmp_path / "speculative_decoding_verification_17_gb300"
    (pkg / "csrc").mkdir(parents=True)
    (tmp_path / "include").mkdir()
    (pkg / "_native.py").write_text('ARCH = ["-gencode", "x"]\nNVCC_FLAGS = ["-O3"]\n')
    (tmp_path / "include" / "api.h").write_text("int f(int);\n")
    unit = pkg / "csrc" / "k.cu"
    unit.write_text('#include "api.h"\n// a kernel\nint f(int x) { return x + 1; }\n')
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.source_digest("k.cu")
    unit.write_text('#include "api.h"\n\n/* the same kernel,\n   reworded */\n'
                    'int f(int x) { return x + 1; }  // unchanged\n')
    assert bench.source_digest("k.cu") == d0
    unit.write_text('#include "api.h"\nint f(int x) { return x + 2; }\n')
    assert bench.source_digest("k.cu") != d0
    unit.write_text('#include "api.h"\n// a kernel\nint f(int x) { return x + 1; }\n')
    (tmp_path / "include" / "api.h").write_text("int f(long);\n")  # an included header
    assert bench.source_digest("k.cu") != d0
    (tmp_path / "include" / "api.h").write_text("int f(int);\n")
    (pkg / "_native.py").write_text('ARCH = ["-gencode", "x"]\nNVCC_FLAGS = ["-O2"]\n')
    assert bench.source_digest("k.cu") != d0


def test_committed_profiles_match_the_current_code():
    # every summary that gives a traffic figure was captured on the code as it stands
    for kernel, workload, unit in [
            ("segment_kernel", "sample_b512_k8_v128256_bf16", "sv_verify.cu"),
            ("segment_kernel", "sample_b256_k4_v151936_f32", "sv_verify.cu"),
            ("segment_kernel", "gate_n1280_v151936_f32", "sv_gate.cu")]:
        assert os.path.exists(os.path.join(bench.ROOT, "profiles", f"{kernel}_{workload}.md"))
        t = bench.profiled_traffic(kernel, workload, unit)
        assert t is not None and t > 0, workload
