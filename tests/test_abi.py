"""CPU tests of the C ABI boundary: the library loads, exports every function
include/kvq.h declares, and its host-side arithmetic and validation behave
as documented.  Nothing here launches a kernel."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def K():
    from quantized_kv_decode_gb300 import build
    build.build()
    import quantized_kv_decode_gb300 as K
    K.lib()
    return K


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("kvq_append", "kvq_decode_attn", "kvq_cache_bytes", "kvq_decode_workspace_size",
              "kvq_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(K):
    lib = ctypes.CDLL(K._lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing
    # the binding declares the same set, with the header's names
    assert sorted(K._lib.SIGNATURES) == declared_functions()


def test_library_exports_nothing_else(K):
    """The library is built with hidden default visibility: its dynamic
    symbol table holds the C ABI and nothing else, so two builds loaded in
    one process (release and debug) share no C++ symbol."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", K._lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    names = sorted(line.split()[-1] for line in out.splitlines() if line.strip())
    assert names == declared_functions()


def test_status_strings(K):
    for st in range(5):
        assert K.kvq_status_string(st).startswith("KVQ_")


def test_cache_bytes_against_page_figures(K, golden):
    """kvq_cache_bytes restates the pages' per-token byte counts."""
    _, rows = golden("fp16_cache_sizes.txt")
    for r in rows:
        layers, kvh, hd, nbytes, tokens, expect, tol = map(int, r[2:9])
        desc = K.make_desc(16, 0, kvh, hd, K.KVQ_DENSE, 1)
        assert abs(layers * K.kvq_cache_bytes(desc, tokens) - expect) <= tol, r[1]
    kv, grp = golden("kvq_byte_accounting.txt")
    L, H, D = kv["layers"], kv["kv_heads"], kv["head_dim"]
    per_tok = L * K.kvq_cache_bytes(K.make_desc(4, 128, H, D, K.KVQ_DENSE, 1), 1)
    assert per_tok == kv["int4_g128_total_per_token_kib"] * 1024
    seq = L * K.kvq_cache_bytes(K.make_desc(4, 128, H, D, K.KVQ_DENSE, 1), kv["seq_tokens"])
    assert seq == kv["int4_g128_seq_mib"] * 2 ** 20
    for r in grp:
        g, eff_bits = int(r[1]), float(r[3])
        b = L * K.kvq_cache_bytes(K.make_desc(4, g, H, D, K.KVQ_DENSE, 1), 1)
        assert abs(b * 8 / (2 * L * H * D) - eff_bits) < 1e-9


def test_cache_array_bytes(K):
    d = K.make_desc(4, 32, 8, 128, K.KVQ_DENSE, 4112)
    codes, hdr = K.kvq_cache_array_bytes(d, 8)
    assert codes == 8 * 8 * 4112 * 64 and hdr == 8 * 8 * 4112 * 4 * 2
    p = K.make_desc(8, 64, 2, 64, K.KVQ_PAGED, 16, 1000, 257)
    codes, hdr = K.kvq_cache_array_bytes(p, 0)
    assert codes == 1000 * 2 * 16 * 64 and hdr == 1000 * 2 * 16 * 1 * 2
    f = K.make_desc(16, 0, 4, 256, K.KVQ_DENSE, 10)
    assert K.kvq_cache_array_bytes(f, 3) == (3 * 4 * 10 * 512, 0)


@pytest.mark.parametrize("field,value", [
    ("bits", 5), ("bits", 3), ("group_size", 12), ("group_size", 0), ("group_size", 48),
    ("num_kv_heads", 0), ("layout", 3), ("capacity", 0), ("head_dim", 100)])
def test_invalid_descriptor_rejected(K, field, value):
    d = K.make_desc(4, 32, 8, 128, K.KVQ_DENSE, 64)
    setattr(d, field, value)
    with pytest.raises(K.KVQError) as e:
        K.kvq_cache_array_bytes(d, 1)
    assert e.value.status == K.KVQ_ERR_INVALID_ARG
    assert K.kvq_cache_bytes(d, 1) == 0


def test_unsupported_head_dim(K):
    d = K.make_desc(4, 32, 8, 512, K.KVQ_DENSE, 64)
    with pytest.raises(K.KVQError) as e:
        K.kvq_cache_array_bytes(d, 1)
    assert e.value.status == K.KVQ_ERR_UNSUPPORTED
    assert K.kvq_cache_bytes(d, 1) == 2 * 8 * (256 + 4 * 16)


def test_append_and_decode_validate_before_launch(K):
    """Host-visible errors return synchronously, before any CUDA call."""
    from ctypes import byref
    lib = K.lib()
    d = K.make_desc(4, 32, 2, 128, K.KVQ_DENSE, 64)
    empty = K.kvq_cache()
    assert lib.kvq_append(byref(d), byref(empty), 1, 1, 16, 16, 16, None, None) == K.KVQ_ERR_INVALID_ARG
    assert lib.kvq_append(None, byref(empty), 1, 1, 16, 16, 16, None, None) == K.KVQ_ERR_INVALID_ARG
    fake = K.kvq_cache(16, 32, 48, 64, 80, 96, None)
    # null inputs
    assert lib.kvq_append(byref(d), byref(fake), 1, 1, None, 16, 16, None, None) == K.KVQ_ERR_INVALID_ARG
    # misaligned input
    assert lib.kvq_append(byref(d), byref(fake), 1, 1, 18, 16, 16, None, None) == K.KVQ_ERR_INVALID_ARG
    # nothing to do is not an error
    assert lib.kvq_append(byref(d), byref(fake), 0, 1, None, None, None, None, None) == K.KVQ_OK
    # heads not a multiple of the KV heads
    assert lib.kvq_decode_attn(byref(d), byref(fake), 1, 3, 16, 16, 64, 1, 0.0, 16, None, 0,
                               None, None) == K.KVQ_ERR_INVALID_ARG
    # too many query heads per KV head for the kernels
    assert lib.kvq_decode_attn(byref(d), byref(fake), 1, 2 * 17, 16, 16, 64, 1, 0.0, 16, None,
                               0, None, None) == K.KVQ_ERR_UNSUPPORTED
    # more sequences than a grid dimension holds
    assert lib.kvq_decode_attn(byref(d), byref(fake), 65536, 2, 16, 16, 64, 1, 0.0, 16, None,
                               0, None, None) == K.KVQ_ERR_UNSUPPORTED
    kd = K.make_desc(4, 32, 2, 128, K.KVQ_DENSE, 64, k_per_channel=True, sink_tokens=4)
    kfake = K.kvq_cache(16, 32, 48, 64, 80, 96, None, 112, 128)
    assert lib.kvq_append(byref(kd), byref(kfake), 65536, 1, 16, 16, 16, None,
                          None) == K.KVQ_ERR_UNSUPPORTED
    # explicit split count needs a workspace
    assert lib.kvq_decode_attn(byref(d), byref(fake), 1, 2, 16, 16, 640, 4, 0.0, 16, None, 0,
                               None, None) == K.KVQ_ERR_WORKSPACE
    # negative scale
    assert lib.kvq_decode_attn(byref(d), byref(fake), 1, 2, 16, 16, 64, 1, -1.0, 16, None, 0,
                               None, None) == K.KVQ_ERR_INVALID_ARG
    # paged without a block table
    p = K.make_desc(4, 32, 2, 128, K.KVQ_PAGED, 16, 10, 4)
    assert lib.kvq_append(byref(p), byref(fake), 1, 1, 16, 16, 16, None, None) == K.KVQ_ERR_INVALID_ARG


def test_explicit_split_counts(K):
    d = K.make_desc(4, 32, 32, 128, K.KVQ_DENSE, 4112)
    assert K.kvq_decode_num_splits(d, 8, 32, 4097, 1) == 1
    assert K.kvq_decode_num_splits(d, 8, 32, 4097, 7) == 7
    # never more splits than 64-token tiles
    assert K.kvq_decode_num_splits(d, 8, 32, 100, 50) == 2
    assert K.kvq_decode_workspace_size(d, 8, 32, 4097, 1) == 0
    ws = K.kvq_decode_workspace_size(d, 8, 32, 4097, 4)
    assert ws >= 8 * 32 * 4 * (128 + 2) * 4


def test_symmetric_descriptor(K):
    """A symmetric cache keeps a 2-byte scale per group and no zero arrays."""
    from ctypes import byref
    d = K.make_desc(4, 32, 8, 128, K.KVQ_DENSE, 64, symmetric=True)
    assert K.kvq_cache_bytes(d, 1) == 2 * 8 * (64 + 2 * 4)
    assert K.kvq_cache_array_bytes(d, 2) == (2 * 8 * 64 * 64, 2 * 8 * 64 * 4 * 2)
    for bad in (K.make_desc(16, 0, 8, 128, K.KVQ_DENSE, 64, symmetric=True),):
        assert K.kvq_cache_bytes(bad, 1) == 0
    d2 = K.make_desc(4, 32, 8, 128, K.KVQ_DENSE, 64)
    d2.symmetric = 2
    assert K.kvq_cache_bytes(d2, 1) == 0
    lib = K.lib()
    no_zero = K.kvq_cache(16, 32, 48, None, 80, None, None)
    # symmetric: the zero arrays are not needed (batch 0: validated, nothing runs)
    assert lib.kvq_append(byref(d), byref(no_zero), 0, 1, None, None, None, None, None) == K.KVQ_OK
    asym = K.make_desc(4, 32, 8, 128, K.KVQ_DENSE, 64)
    assert lib.kvq_append(byref(asym), byref(no_zero), 0, 1, None, None, None, None,
                          None) == K.KVQ_ERR_INVALID_ARG


def test_axis_aware_descriptor(K):
    """Byte accounting of axis-aware caches equals the oracle's, and the
    descriptor rules are enforced on the host."""
    import oracle as O
    for (bits, g, S, D, H) in ((4, 32, 4, 128, 8), (8, 64, 0, 128, 2), (4, 16, 3, 64, 4)):
        d = K.make_desc(bits, g, H, D, K.KVQ_DENSE, 4 * g, k_per_channel=True, sink_tokens=S)
        for tokens in (0, 1, S, S + g - 1, S + g, S + 3 * g + 5, 1000):
            assert K.kvq_cache_bytes(d, tokens) == O.kivi_cache_bytes(H, D, tokens, bits, g, S)
        assert K.kvq_cache_window_bytes(d, 3) == 3 * H * (S + g) * D * 2
        codes, hdr = K.kvq_cache_array_bytes(d, 2)
        assert codes == 2 * H * 4 * g * D * bits // 8 and hdr == 2 * H * 4 * g * (D // g) * 2
    assert K.kvq_cache_window_bytes(K.make_desc(4, 32, 8, 128, K.KVQ_DENSE, 64), 3) == 0
    # paged: pages of the quantized region hold whole blocks; the arrays are
    # per page (K headers: page_size / g blocks of D channels per page)
    pd = K.make_desc(4, 32, 8, 128, K.KVQ_PAGED, 64, 10, 4, k_per_channel=True, sink_tokens=4)
    codes, hdr = K.kvq_cache_array_bytes(pd, 1)
    assert codes == 10 * 8 * 64 * 64 and hdr == 10 * 8 * (64 // 32) * 128 * 2
    assert K.kvq_cache_bytes(K.make_desc(4, 32, 8, 128, K.KVQ_PAGED, 48, 10, 4,
                                         k_per_channel=True), 1) == 0
    bad = [dict(symmetric=True), dict(sink_tokens=-1), dict(sink_tokens=64)]
    for kw in bad:
        d = K.make_desc(4, 32, 8, 128, K.KVQ_DENSE, 64, k_per_channel=True, **kw)
        assert K.kvq_cache_bytes(d, 1) == 0, kw
    assert K.kvq_cache_bytes(K.make_desc(4, 32, 8, 128, K.KVQ_DENSE, 48, k_per_channel=True), 1) == 0
    assert K.kvq_cache_bytes(K.make_desc(16, 0, 8, 128, K.KVQ_DENSE, 64, k_per_channel=True), 1) == 0
    assert K.kvq_cache_bytes(K.make_desc(4, 32, 8, 128, K.KVQ_DENSE, 64, sink_tokens=2), 1) == 0


def test_lowbit_descriptors(K):
    """INT2 packs four codes per byte; NF4 keeps a 2-byte scale per group and
    no zero arrays; NF4 requires bits 4 and excludes the symmetric and
    axis-aware options."""
    import oracle as O
    d2 = K.make_desc(2, 32, 8, 128, K.KVQ_DENSE, 64)
    assert K.kvq_cache_bytes(d2, 1) == O.kv_cache_bytes(1, 8, 128, 1, 2, 32) == 2 * 8 * (32 + 16)
    assert K.kvq_cache_array_bytes(d2, 1)[0] == 8 * 64 * 32
    dn = K.make_desc(4, 64, 8, 128, K.KVQ_DENSE, 64, nf4=True)
    assert K.kvq_cache_bytes(dn, 1) == O.kv_cache_bytes(1, 8, 128, 1, 4, 64, nf4=True)
    for kw in (dict(bits=8), dict(bits=2), dict(symmetric=True)):
        args = dict(bits=4, symmetric=False)
        args.update(kw)
        d = K.make_desc(args["bits"], 64, 8, 128, K.KVQ_DENSE, 64, symmetric=args["symmetric"], nf4=True)
        assert K.kvq_cache_bytes(d, 1) == 0, kw
    assert K.kvq_cache_bytes(K.make_desc(4, 64, 8, 128, K.KVQ_DENSE, 64, k_per_channel=True,
                                         nf4=True), 1) == 0
    assert K.kvq_cache_bytes(K.make_desc(2, 32, 8, 128, K.KVQ_DENSE, 64, k_per_channel=True), 1) == 0


def test_release_library_has_no_debug_checks(K):
    """The release library reports no bounds checks and refuses the
    debug-only extent control (host functions, no launch)."""
    lib = K._lib.load(K._lib.LIB_PATH)
    assert lib.kvq_debug_checks() == 0
    assert lib.kvq_debug_shrink_extent(K._lib.KVQ_ARRAY_K_CODES, 16) == K.KVQ_ERR_UNSUPPORTED
    assert K._lib.KVQ_ARRAY_WORKSPACE == 14   # the header's kvq_array order
    text = open(HEADER).read()
    ids = dict((m.group(1), int(m.group(2)))
               for m in re.finditer(r"(KVQ_ARRAY_\w+)\s*=\s*(\d+)", text))
    assert ids == {n: getattr(K._lib, n) for n in ids if n != "KVQ_ARRAY_COUNT"} | \
        {"KVQ_ARRAY_COUNT": 15}
