"""The workspace-free attention entry point, for callers that cannot allocate
device memory (a host whose device memory is all owned by its own pool, a
serving loop that must not call cudaMalloc because it synchronises the
device, a binding without an allocator).  It must give the same output as the
regular entry point, call after call, while reusing its fixed device scratch.

Collected last on purpose (file name): a failure here never hides the other
tests' results when pytest stops at the first failure.
"""
import numpy as np
import pytest

import synth
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_variable_gb300 import build
    build.build()


def _cases():
    # a decode batch whose long sequences are split (the scratch holds the
    # split-KV partials) and a mixed prefill/decode batch
    rng = np.random.default_rng(77)
    dec = synth.make_case(synth.uniform_spec("noalloc-decode", 8, 1, 5000, hq=32, hkv=8, d=128, page_size=16), rng)
    mixed = H.gpu_random_case(78, page_size=16, max_cache=900, max_new=60)
    return [dec, mixed]


@pytest.mark.parametrize("idx", [0, 1])
def test_noalloc_matches_workspace_entry_point(idx):
    import torch
    case = _cases()[idx]
    g = H.GpuCase(case)                        # one CTA per SM: the long decode units are split
    g.run()
    assert g.status() == 0
    want = g.out.clone()
    if idx == 0:
        assert g.plan.stats()["num_split_units"] > 0
    for _ in range(2):                          # two calls in a row share the scratch
        g.out.fill_(float("nan"))
        g.pkv.attn_varlen_kvcache_fwd_noalloc(g.problem, g.args(), g.plan)
        torch.cuda.synchronize()
        assert g.pkv.get_status_noalloc() == 0, g.pkv.last_error()
        H.compare_out(g.out, H.bf16_to_f64(want), H.BF16_TOL, what="noalloc out")


def test_noalloc_device_status_is_readable():
    """A device-side error of a workspace-free call (a block_table entry past
    the page pool, which the kernels skip instead of reading) shows in the
    status word of the fixed scratch; the next good call clears it."""
    case = synth.config1()
    g = H.GpuCase(case)
    bad = g.block_table.clone()
    bad[0, 1] = 10_000
    good_table = g.block_table
    g.block_table = bad
    g.pkv.attn_varlen_kvcache_fwd_noalloc(g.problem, g.args(), g.plan)
    assert g.pkv.get_status_noalloc() == 6      # PKV_ERR_DEVICE_BOUNDS
    assert g.pkv.get_status_noalloc() == 0      # reading resets it
    g.block_table = good_table
    g.pkv.attn_varlen_kvcache_fwd_noalloc(g.problem, g.args(), g.plan)
    assert g.pkv.get_status_noalloc() == 0
