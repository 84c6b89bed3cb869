"""GPU tests of kvq_decode_attn_static_ws, the decode entry point that takes
its split scratch from a static array in the library instead of a caller
workspace.

It is called straight through the C ABI (ctypes, caller-made buffers only)
and compared with kvq_decode_attn on the same inputs: two calls in a row
must each agree within the decode tolerance (max |err| <= 2e-3, relative L2
<= 1e-3), and the second call must leave the device's free memory as the
first left it.  The cases force several splits so that the static scratch is
really used.  A request whose workspace would exceed the array is rejected
before any launch, and the planner's scratch for every benchmark workload
fits the array.  The file is named to be collected last and its tests also
pass alone in a fresh process.
"""
import os
import re
from ctypes import byref

import numpy as np
import pytest

from tests._cases import Case, assert_close, make_inputs, run_gpu
from tests.conftest import ROOT

pytestmark = pytest.mark.gpu


def _static_bytes():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    m = re.search(r"#define\s+KVQ_STATIC_WORKSPACE_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    return int(m.group(1)) << int(m.group(2))


def _call_static(K, cache, q, seq_lens, max_seq_len, out, status, num_splits):
    import torch
    return K.lib().kvq_decode_attn_static_ws(
        byref(cache.desc), byref(cache.ptrs), q.shape[0], q.shape[1], q.data_ptr(),
        seq_lens.data_ptr(), int(max_seq_len), int(num_splits), 0.0, out.data_ptr(),
        status.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("case,splits", [
    (Case(B=3, Hq=8, Hkv=2, D=128, bits=4, g=32, lens=np.array([700, 0, 451]), seed=41), 4),
    (Case(B=2, Hq=4, Hkv=4, D=128, bits=8, g=64, lens=np.array([1200, 333]), seed=42), 7),
    (Case(B=4, Hq=16, Hkv=1, D=128, bits=4, g=16, lens=np.array([90, 600, 1, 250]), seed=43), 3),
    (Case(B=5, Hq=14, Hkv=2, D=64, bits=4, g=32, lens=np.array([130, 1, 64, 47, 300]), seed=44,
          layout="paged", page_size=16), 2),
])
def test_static_scratch_matches_workspace_entry_point(case, splits):
    import torch
    import quantized_kv_decode_gb300 as K
    inp = make_inputs(case)
    ref = run_gpu(case, inp, num_splits=splits)       # cache filled, then kvq_decode_attn
    assert ref["status"] == 0
    cache = ref["cache"]
    dev = "cuda"
    q = torch.from_numpy(inp["q"]).to(dev)
    seq_lens = torch.from_numpy(case.lens.astype(np.int32) + 1).to(dev)
    max_len = inp["Lctx"] + 1
    assert K.kvq_decode_workspace_size(cache.desc, case.B, case.Hq, max_len, splits) > 0
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = [torch.full_like(q, float("nan")) for _ in range(2)]
    free = []
    for out in outs:                                    # two calls in a row
        st = _call_static(K, cache, q, seq_lens, max_len, out, status, splits)
        assert st == K.KVQ_OK, K.kvq_status_string(st)
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        assert int(status.item()) == 0
        assert_close(out.cpu().numpy(), ref["out"].astype(np.float64))
    # after the first call (which may load the library's device code), a call
    # takes no device memory: the free bytes the driver reports do not move
    assert free[1] == free[0]


def test_static_scratch_rejects_oversized_request():
    """A split count whose partials exceed the static array is refused with
    KVQ_ERR_WORKSPACE before anything runs; the output stays untouched."""
    import torch
    import quantized_kv_decode_gb300 as K
    dev = "cuda"
    B, Hq, Hkv, D, L = 64, 32, 8, 128, 2048
    desc = K.make_desc(4, 32, Hkv, D, K.KVQ_DENSE, L)
    cache = K.KVCache.allocate(desc, B, dev)
    splits = 16
    assert K.kvq_decode_workspace_size(desc, B, Hq, L, splits) > _static_bytes()
    q = torch.zeros((B, Hq, D), dtype=torch.float16, device=dev)
    seq_lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    out = torch.full_like(q, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = _call_static(K, cache, q, seq_lens, L, out, status, splits)
    assert st == K.KVQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and int(status.item()) == 0
    # the same request with the planner's own split count fits and runs
    assert K.kvq_decode_workspace_size(desc, B, Hq, L, 0) <= _static_bytes()
    assert _call_static(K, cache, q, seq_lens, L, out, status, 0) == K.KVQ_OK
    torch.cuda.synchronize()
    assert not bool(torch.isnan(out).any())


def test_static_scratch_covers_the_workloads():
    """The planner's split scratch for each benchmark workload's full shape
    (automatic split choice) fits the static array."""
    import quantized_kv_decode_gb300 as K
    from quantized_kv_decode_gb300 import synth
    for name, bits in (("tiny", 4), ("mha7b", 4), ("mha7b", 16), ("gqa_mix", 4), ("long", 4),
                       ("long", 8), ("paged", 4)):
        w = synth.WORKLOADS[name]
        L = w.ctx[1] + 1
        if w.layout == "paged":
            pages = -(-L // w.page_size)
            desc = K.make_desc(bits, w.group_size, w.num_kv_heads, w.head_dim, K.KVQ_PAGED,
                               w.page_size, pages * w.batch, pages)
        else:
            desc = K.make_desc(bits, w.group_size if bits != 16 else 0, w.num_kv_heads,
                               w.head_dim, K.KVQ_DENSE, (L + 15) // 16 * 16)
        need = K.kvq_decode_workspace_size(desc, w.batch, w.num_q_heads, L, 0)
        assert need <= _static_bytes(), (name, bits, need)
