"""The Python binding on a machine without a GPU: it refuses host tensors and
wrong dtypes or layouts with an error before calling the library, so there is
no silent CPU path; the enum values and the status text match the header."""
import re
import os

import pytest
import torch

import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    vit.lib()


def _qkv(T=8, H=2, D=32, device="cpu", dtype=torch.bfloat16):
    return [torch.zeros((T, H, D), dtype=dtype, device=device) for _ in range(3)]


def test_host_tensors_are_refused_not_computed():
    q, k, v = _qkv()
    cu = torch.tensor([0, 8], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        vit.varlen_attn(q, k, v, cu, 8)
    pos = torch.zeros((8, 2), dtype=torch.int32)
    inv = torch.zeros(8, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA"):
        vit.qk_norm_rope(q, k, pos, inv)
    with pytest.raises(ValueError):
        vit.rope_freqs(torch.tensor([[2, 4]], dtype=torch.int32), 8, 32)
    with pytest.raises(ValueError):
        vit.rope_table(inv, 32, 4)
    with pytest.raises(ValueError):
        vit.varlen_attn_padded(q, k, v, torch.zeros(1, dtype=torch.int32), torch.full((1,), 8, dtype=torch.int32), 8)


def test_wrong_dtype_and_layout_are_refused():
    q, k, v = _qkv(dtype=torch.float16)
    with pytest.raises(ValueError):
        vit.varlen_attn(q, k, v, None, 8, num_segments=1)
    q, k, v = _qkv()
    with pytest.raises(ValueError):                                   # head stride must be D
        vit.varlen_attn(q.transpose(1, 2), k, v, None, 8, num_segments=1)
    with pytest.raises(ValueError):
        vit.varlen_attn(q, k, v, None, 8)                             # no cu_seqlens and no count
    with pytest.raises(ValueError):
        vit.qk_norm_rope(None, None, torch.zeros((8, 2), dtype=torch.int32), torch.zeros(8))


def test_enums_match_the_header():
    text = open(os.path.join(ROOT, "include", "vit_attn.h")).read()
    assert int(re.search(r"VIT_ROPE_ROTATE_HALF\s*=\s*(\d+)", text).group(1)) == vit.ROPE_ROTATE_HALF
    assert int(re.search(r"VIT_ROPE_INTERLEAVED\s*=\s*(\d+)", text).group(1)) == vit.ROPE_INTERLEAVED
    assert int(re.search(r"#define VIT_MAX_SEGMENTS\s+(\d+)", text).group(1)) == vit.MAX_SEGMENTS
    codes = {m.group(1): int(m.group(2)) for m in re.finditer(r"(VIT_ERR_\w+)\s*=\s*(-\d+)", text)}
    assert codes["VIT_ERR_POSITION_RANGE"] == -15 and len(codes) == 15
    for name, code in codes.items():
        assert vit.status_string(code) != "unknown status", name
    err = vit.VitError(codes["VIT_ERR_BAD_SEQLENS"], "call")
    assert err.code == -10 and "cu_seqlens" in str(err)
