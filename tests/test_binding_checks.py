"""CPU tests of the Python binding's buffer checks (no GPU: tensors are stand-ins that
report CUDA placement; the check only reads their sizes and addresses)."""

import pytest
import torch

from collective_datapath_copy_gb300 import _lib
from collective_datapath_copy_gb300.plan import _check_buffers


class OnDevice:
    """A CPU tensor that answers like a CUDA tensor for the binding's checks."""

    def __init__(self, t):
        self.t = t

    is_cuda = True

    @property
    def nbytes(self):
        return self.t.nbytes

    def is_contiguous(self):
        return self.t.is_contiguous()

    def data_ptr(self):
        return self.t.data_ptr()

    def untyped_storage(self):
        return self.t.untyped_storage()


def check(ts, nbytes, stride=0, count=1):
    _check_buffers(len(ts), ts, [True] * len(ts), nbytes, stride, count, "test")


def test_buffers_that_hold_the_run_pass():
    a = OnDevice(torch.zeros(1024, dtype=torch.int16))
    check([a], [2048])
    check([a], [1024], stride=512, count=3)          # 2 x 512 + 1024 = 2048
    big = torch.zeros(3, 512, dtype=torch.int16)
    check([OnDevice(big[0])], [1024], stride=1024, count=3)   # the view's storage holds it
    check([OnDevice(big[2])], [1024], stride=-1024, count=3)  # negative strides reach back


def test_buffers_too_small_are_rejected_with_ebounds():
    a = OnDevice(torch.zeros(1024, dtype=torch.int16))
    for kw in (dict(nbytes=[2050]), dict(nbytes=[1024], stride=1024, count=3)):
        with pytest.raises(_lib.CollError) as e:
            check([a], kw.pop("nbytes"), **kw)
        assert e.value.code == _lib.D["COLL_EBOUNDS"]
    big = torch.zeros(3, 512, dtype=torch.int16)
    with pytest.raises(_lib.CollError):
        check([OnDevice(big[1])], [1024], stride=1024, count=3)   # past the storage's end
    with pytest.raises(_lib.CollError):
        check([OnDevice(big[0])], [1024], stride=-1024, count=2)  # before its start


def test_host_tensors_and_unused_ranks():
    with pytest.raises(ValueError):
        check([torch.zeros(4)], [8])
    # ranks the run does not touch are not checked, missing buffers are left to the library
    _check_buffers(2, [None, torch.zeros(1)], [True, False], [8, 8], 0, 1, "test")
