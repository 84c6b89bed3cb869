"""GPU tests of the debug build (libkvq_debug.so, compiled with KVQ_DEBUG).

In that build every global load and store of the kernels is first checked
against the byte extent of the caller array it addresses; an access outside
is skipped and flags KVQ_FLAG_OOB.  These tests route the binding to the
debug library and

  * run one case of every kernel path (both append kernels, the tensor-core
    decode kernel in each score layout and format, dense and paged, fused
    and split, the CUDA-core and per-element kernels, the split merge, the
    axis-aware append inside and outside the decode launch, the static-
    workspace entry point) against the oracle: the results agree, no check
    fires, and the guard bytes around every array stay intact;
  * shorten one array's extent at a time (kvq_debug_shrink_extent) below
    what the call touches and check that the checks fire: KVQ_FLAG_OOB is
    set and nothing is written outside the arrays.  The shortened part still
    lies inside the caller's allocation, so no access leaves it.
"""
import numpy as np
import pytest

from tests._cases import Case, assert_close, make_inputs, oracle_step, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib():
    from quantized_kv_decode_gb300 import _lib, build
    handle = _lib.load(build.build(debug=True))
    assert handle.kvq_debug_checks() == 1
    prev = _lib.use(handle)
    try:
        yield handle
    finally:
        for a in range(15):
            handle.kvq_debug_shrink_extent(a, 0)
        _lib.use(prev)


def _lens(*xs):
    return np.array(xs)


# one case per kernel path (run_gpu: kvq_append populates, then the step)
PATHS = [
    ("mha_int4_token_rows_fused", Case(B=3, Hq=4, Hkv=4, D=128, bits=4, g=32, lens=_lens(300, 31, 97), seed=1), 0, True),
    ("mha_int4_splits", Case(B=2, Hq=4, Hkv=4, D=128, bits=4, g=32, lens=_lens(700, 45), seed=2), 3, False),
    ("gqa_16_columns", Case(B=3, Hq=16, Hkv=4, D=128, bits=4, g=32, lens=_lens(260, 0, 33), seed=3), 0, True),
    ("gqa_8_columns_int8", Case(B=2, Hq=8, Hkv=2, D=128, bits=8, g=64, lens=_lens(200, 75), seed=4), 2, True),
    ("paged_g7_d64", Case(B=4, Hq=14, Hkv=2, D=64, bits=4, g=32, lens=_lens(130, 1, 64, 300), seed=5,
                          layout="paged", page_size=16), 0, True),
    ("paged_splits", Case(B=2, Hq=8, Hkv=2, D=128, bits=4, g=32, lens=_lens(500, 90), seed=6,
                          layout="paged", page_size=32), 3, False),
    ("symmetric", Case(B=2, Hq=8, Hkv=8, D=128, bits=4, g=32, lens=_lens(150, 60), seed=7, symmetric=True), 0, True),
    ("nf4", Case(B=2, Hq=8, Hkv=2, D=128, bits=4, g=64, lens=_lens(180, 20), seed=8, nf4=True), 0, True),
    ("int2", Case(B=2, Hq=4, Hkv=4, D=128, bits=2, g=32, lens=_lens(170, 9), seed=9), 0, True),
    ("cuda_core_g8", Case(B=2, Hq=8, Hkv=2, D=128, bits=4, g=8, lens=_lens(120, 40), seed=10), 2, False),
    ("fp16_tensor_core", Case(B=2, Hq=4, Hkv=2, D=128, bits=16, g=0, lens=_lens(90, 33), seed=11), 0, True),
    ("cuda_core_fp16_d256", Case(B=2, Hq=2, Hkv=1, D=256, bits=16, g=0, lens=_lens(60, 21), seed=13), 2, False),
    ("cuda_core_g16_heads", Case(B=2, Hq=32, Hkv=2, D=64, bits=8, g=32, lens=_lens(77, 140), seed=12), 0, False),
]


@pytest.mark.parametrize("name,case,splits,fused", PATHS, ids=[p[0] for p in PATHS])
def test_debug_build_paths_clean(debug_lib, name, case, splits, fused):
    inp = make_inputs(case)
    run = run_gpu(case, inp, num_splits=splits, fused=fused)   # guard bytes checked inside
    assert run["status"] == 0, hex(run["status"])             # no KVQ_FLAG_OOB, nothing else
    ref, _ = oracle_step(case, inp)
    assert_close(run["out"], ref)


def test_debug_build_static_workspace_clean(debug_lib):
    import torch
    import quantized_kv_decode_gb300 as K
    from tests.test_zz_no_alloc import _call_static
    case = Case(B=3, Hq=8, Hkv=2, D=128, bits=4, g=32, lens=_lens(700, 0, 451), seed=41)
    inp = make_inputs(case)
    ref = run_gpu(case, inp, num_splits=4)
    q = torch.from_numpy(inp["q"]).cuda()
    lens = torch.from_numpy(case.lens.astype(np.int32) + 1).cuda()
    out = torch.full_like(q, float("nan"))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call_static(K, ref["cache"], q, lens, inp["Lctx"] + 1, out, st, 4) == K.KVQ_OK
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(out.cpu().numpy(), ref["out"].astype(np.float64))


@pytest.mark.parametrize("layout,splits", [("dense", 0), ("dense", 3), ("paged", 0)])
def test_debug_build_axis_aware_clean(debug_lib, layout, splits):
    """Axis-aware caches: the block and window append kernels, the fused step
    (in the decode launch with one split, by the step kernel otherwise), the
    tensor-core kernel's window pass; results as in the release tests."""
    import torch
    import quantized_kv_decode_gb300 as K
    from tests.test_gpu_kivi import _compare_cache, _oracle_out, _paged_kivi_pair, _run
    g, S = 32, 4
    lens = [S + 2 * g - 1, S + 5, 150]
    if layout == "dense":
        K_, cache, k16, v16, q16, kt, vt, q, lt, st = _run(4, g, S, 128, 8, 2, lens, [16, 1],
                                                           splits=splits, seed=5)
        kn = torch.stack([kt[b, L] for b, L in enumerate(lens)]).contiguous()
        vn = torch.stack([vt[b, L] for b, L in enumerate(lens)]).contiguous()
    else:
        pair = _paged_kivi_pair(K, 4, 4, g, 128, lens, seed=9)
        cache, k16, v16, q16 = pair["paged"], pair["k16"], pair["v16"], pair["q16"]
        kn, vn, S = pair["kn"], pair["vn"], pair["S"]
        q = torch.from_numpy(q16).cuda()
        lt = torch.tensor(lens, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = K.kvq_append_decode_attn(cache, kn, vn, q, lt, max(lens) + 1, dev_status=st,
                                   num_splits=splits)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, hex(int(st.item()))
    lens1 = [L + 1 for L in lens]
    if layout == "dense":
        _compare_cache(cache, k16, v16, lens1, 4, g, S)
    assert_close(out.cpu().numpy(), _oracle_out(q16, k16, v16, lens1, 4, g, S))


def _shrunk_run(handle, array, nbytes, case, splits=0, fused=False):
    try:
        assert handle.kvq_debug_shrink_extent(array, nbytes) == 0
        return run_gpu(case, make_inputs(case), num_splits=splits, fused=fused)
    finally:
        handle.kvq_debug_shrink_extent(array, 0)


DENSE = Case(B=2, Hq=8, Hkv=4, D=128, bits=4, g=32, lens=_lens(200, 150), seed=21)
PAGED = Case(B=2, Hq=14, Hkv=2, D=64, bits=4, g=32, lens=_lens(90, 120), seed=22, layout="paged",
             page_size=16)
CC = Case(B=2, Hq=4, Hkv=2, D=128, bits=4, g=8, lens=_lens(100, 60), seed=23)


@pytest.mark.parametrize("array,frac,case,splits,fused", [
    ("KVQ_ARRAY_K_CODES", 0.5, DENSE, 0, False),
    ("KVQ_ARRAY_V_CODES", 0.5, DENSE, 0, True),
    ("KVQ_ARRAY_K_SCALE", 0.5, DENSE, 0, False),
    ("KVQ_ARRAY_V_ZERO", 0.5, DENSE, 0, True),
    ("KVQ_ARRAY_Q", 0.5, DENSE, 0, False),
    ("KVQ_ARRAY_OUT", 0.5, DENSE, 0, False),
    ("KVQ_ARRAY_SEQ_LENS", 0.5, DENSE, 0, True),
    ("KVQ_ARRAY_K_NEW", 0.5, DENSE, 0, True),
    ("KVQ_ARRAY_WORKSPACE", 1.0, DENSE, 3, False),
    ("KVQ_ARRAY_BLOCK_TABLE", 0.5, PAGED, 0, True),
    ("KVQ_ARRAY_V_CODES", 0.5, PAGED, 0, False),
    ("KVQ_ARRAY_K_CODES", 0.5, CC, 2, False),
    ("KVQ_ARRAY_V_SCALE", 0.5, CC, 0, False),
])
def test_debug_checks_fire_on_a_short_extent(debug_lib, array, frac, case, splits, fused):
    """With one array's extent cut below what the call touches, the checks
    skip the accesses to the cut part and flag KVQ_FLAG_OOB; the guard bytes
    around every array stay intact (run_gpu asserts that)."""
    import quantized_kv_decode_gb300 as K
    from quantized_kv_decode_gb300 import _lib
    a = getattr(_lib, array)
    inp = make_inputs(case)
    clean = run_gpu(case, inp, num_splits=splits, fused=fused)
    assert clean["status"] == 0
    # the array's size for this call, from the same rules the host uses
    sizes = _call_sizes(K, case, clean, splits)
    cut = max(4, int(sizes[array] * frac)) // 4 * 4
    run = _shrunk_run(debug_lib, a, cut, case, splits=splits, fused=fused)
    assert run["status"] & K.KVQ_FLAG_OOB, hex(run["status"])


def _call_sizes(K, case, run, splits):
    desc = run["desc"]
    lmax = int(case.lens.max()) + 1
    cb, hb = K.kvq_cache_array_bytes(desc, case.B)
    qb = case.B * case.Hq * case.D * 2
    return {
        "KVQ_ARRAY_K_CODES": cb, "KVQ_ARRAY_V_CODES": cb,
        "KVQ_ARRAY_K_SCALE": hb, "KVQ_ARRAY_V_SCALE": hb, "KVQ_ARRAY_K_ZERO": hb,
        "KVQ_ARRAY_V_ZERO": hb,
        "KVQ_ARRAY_Q": qb, "KVQ_ARRAY_OUT": qb,
        "KVQ_ARRAY_SEQ_LENS": case.B * 4,
        "KVQ_ARRAY_K_NEW": case.B * case.Hkv * case.D * 2,
        "KVQ_ARRAY_WORKSPACE": K.kvq_decode_workspace_size(desc, case.B, case.Hq, lmax, splits),
        "KVQ_ARRAY_BLOCK_TABLE": case.B * desc.max_blocks_per_seq * 4,
    }


def test_release_and_debug_builds_in_one_process(debug_lib):
    """Both builds loaded in one process keep their own kernel set-up: calls
    alternate between them (each library's first call on a shape sets its
    own shared-memory attribute), every call succeeds, each build repeats
    its own output bit for bit, and both match the reference run."""
    import torch
    import quantized_kv_decode_gb300 as K
    from quantized_kv_decode_gb300 import _lib
    release = _lib.load(_lib.LIB_PATH)
    assert release.kvq_debug_checks() == 0
    case = Case(B=3, Hq=12, Hkv=4, D=128, bits=4, g=32, lens=_lens(333, 7, 120), seed=31)
    inp = make_inputs(case)
    ref = run_gpu(case, inp)                        # debug library (the fixture routes to it)
    q = torch.from_numpy(inp["q"]).cuda()
    lens = torch.from_numpy(case.lens.astype(np.int32) + 1).cuda()
    outs = []
    for handle in (release, debug_lib, release, debug_lib):
        prev = _lib.use(handle)
        try:
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            outs.append(K.kvq_decode_attn(ref["cache"], q, lens, inp["Lctx"] + 1, dev_status=st))
            torch.cuda.synchronize()
            assert int(st.item()) == 0
        finally:
            _lib.use(prev)
    assert torch.equal(outs[0], outs[2]) and torch.equal(outs[1], outs[3])
    for o in outs[:2]:
        assert_close(o.cpu().numpy(), ref["out"].astype(np.float64))
