"""Host-side argument checks of the Python binding: they run before any
device pointer is taken, so CPU tensors and a stand-in map exercise them
without a GPU."""
import types

import pytest
import torch

import sparse_voxel_convolution_coord_b300 as sc


def fake_map(n):
    return types.SimpleNamespace(n=n, ptr=1, device=torch.device("cpu"))


def args(n=10, cin=16, cout=32, dt=torch.bfloat16):
    return (torch.zeros(n, cin, dtype=dt), torch.zeros(27, cin, cout, dtype=dt),
            torch.zeros(cout))


@pytest.mark.parametrize("fn", [sc.sc_forward, sc.sc_forward_ex])
def test_operand_checks(fn):
    f, w, b = args()
    with pytest.raises(ValueError, match="same dtype"):
        fn(fake_map(10), f, w.float(), b)
    with pytest.raises(ValueError, match="dtype must be"):
        fn(fake_map(10), f.double(), w.double(), b)
    with pytest.raises(ValueError, match=r"\[27, cin, cout\]"):
        fn(fake_map(10), f, w[:26], b)
    with pytest.raises(ValueError, match="rows, the map"):
        fn(fake_map(11), f, w, b)
    with pytest.raises(ValueError, match="bias must be fp32"):
        fn(fake_map(10), f, w, b.double())


def test_epilogue_checks():
    f, w, b = args()
    m = fake_map(10)
    with pytest.raises(ValueError, match="act must be"):
        sc.sc_forward_ex(m, f, w, b, act="gelu")
    with pytest.raises(ValueError, match="out_dtype must be"):
        sc.sc_forward_ex(m, f, w, b, out_dtype=torch.float64)
    with pytest.raises(ValueError, match="residual must be"):
        sc.sc_forward_ex(m, f, w, b, residual=torch.zeros(10, 32), out_dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out must be"):
        sc.sc_forward_ex(m, f, w, b, out=torch.zeros(10, 32), out_dtype=torch.float16)


def test_device_pointer_check():
    f, w, b = args()
    # every argument valid but on the host: refused before the library is called
    with pytest.raises(ValueError, match="CUDA tensor"):
        sc.sc_forward_ex(fake_map(10), f, w, b)
