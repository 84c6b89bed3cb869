"""The guard bytes the GPU tests put around every array catch a write that
lands outside the array (checked here on the CPU with a planted stray
write), and leave a write inside it unnoticed."""
import pytest

from tests._cases import Guarded, check_guards


@pytest.mark.parametrize("shape,dtype_name", [((3, 5), "float16"), ((7,), "uint8"),
                                              ((2, 3, 4), "int32")])
def test_guards_catch_stray_writes(shape, dtype_name):
    import torch
    dtype = getattr(torch, dtype_name)
    g = Guarded(shape, dtype, "cpu")
    assert g.tensor.shape == shape and g.tensor.dtype == dtype
    assert bool((g.tensor == 0).all())
    g.tensor.fill_(1)                      # every byte of the array itself
    check_guards({"a": g}, "inside")
    for pos in (g.PAD - 1, g.PAD + g.nbytes):  # one byte before, one byte after
        h = Guarded(shape, dtype, "cpu")
        h.buf[pos] = 0
        with pytest.raises(AssertionError, match="outside"):
            check_guards({"a": h}, "planted")
