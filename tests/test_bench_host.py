"""Host logic of the benchmark (no GPU): the kernel-code hash that decides
whether a stored ncu traffic figure belongs to the built kernels, and the
algorithmic work the roofline numbers divide by."""
import numpy as np

import bench
import synth


def test_code_only_drops_comments_keeps_literals():
    src = ('int a = 1;  // note\n'
           '/* block\n   comment */ const char* s = "x // y /* z */";\n'
           "char q = '\"'; char e = '\\\\';\n"
           '\n'
           '   // only a comment\n'
           'int b;\n')
    assert bench._code_only(src) == ('int a = 1;\n'
                                     ' const char* s = "x // y /* z */";\n'
                                     "char q = '\"'; char e = '\\\\';\n"
                                     'int b;')


def test_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "paged_kv_variable_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("__global__ void k(int* p) { p[0] = 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    (csrc / "k.cu").write_text("// a kernel\n__global__ void k(int* p) { p[0] = 1; }  // one store\n\n")
    assert bench.kernel_source_hash() == h0
    (csrc / "k.cu").write_text("__global__ void k(int* p) { p[0] = 2; }\n")
    assert bench.kernel_source_hash() != h0


def test_step_work_counts_attended_pairs():
    """Algorithmic flops: 4 D Hq per attended (query, key) pair, the causal
    count being the bottom-right triangle on top of the cached prefix."""
    spec = synth.config3(True, draw_values=False).spec
    w = bench.step_work(spec)
    lq, lc = 512, 1536
    pairs = lq * lc + lq * (lq + 1) // 2
    assert w["flops"] == 4 * spec.d * spec.hq * spec.batch * pairs
    ncspec = synth.config3(False, draw_values=False).spec
    assert bench.step_work(ncspec)["flops"] == 4 * spec.d * spec.hq * spec.batch * lq * (lq + lc)
