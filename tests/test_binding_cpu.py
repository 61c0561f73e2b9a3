"""The Python binding on a machine without a GPU: every call refuses host tensors
before anything is launched (there is no CPU fallback), an unsupported dtype is
refused, and a missing library is reported loudly."""

import pytest
import torch

import gated_deltanet_tree_gdn_gb300 as gt
from gated_deltanet_tree_gdn_gb300 import _binding


def _host_inputs(B=2, N=8, Hqk=1, Hv=2, d=16, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(0)
    return dict(q=torch.randn(B, N, Hqk, d, generator=g).to(dtype),
                k=torch.randn(B, N, Hqk, d, generator=g).to(dtype),
                v=torch.randn(B, N, Hv, d, generator=g).to(dtype),
                log_alpha=-torch.rand(B, N, Hv, generator=g),
                beta=torch.rand(B, N, Hv, generator=g),
                parent=torch.arange(-1, N - 1, dtype=torch.int32).repeat(B, 1),
                S0=torch.zeros(B, Hv, d, d))


def test_host_tensors_are_refused_without_a_fallback():
    x = _host_inputs()
    with pytest.raises(ValueError, match="CUDA tensor"):
        gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"])
    with pytest.raises(ValueError, match="CUDA tensor"):
        gt.verify_recurrent(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"],
                            x["S0"])
    path = torch.zeros(2, 3, dtype=torch.int32)
    plen = torch.zeros(2, dtype=torch.int32)
    U = torch.zeros(2, 2, 8, 16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        gt.commit(path, plen, U, x["k"], x["log_alpha"], x["S0"])
    with pytest.raises(ValueError, match="CUDA tensor"):
        gt.build_topw(torch.zeros(2, 8, 4), 4, 8)


def test_unsupported_dtype_is_refused():
    with pytest.raises(TypeError):
        _binding._dtype_code(torch.zeros(1, dtype=torch.float16))


def test_missing_library_is_reported(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        _binding.load(str(tmp_path / "libgdntree_missing.so"))
