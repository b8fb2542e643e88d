"""The Python binding on a machine without a GPU: it refuses CPU tensors and
a missing library instead of computing anything on the host (there is no
fallback path)."""
import pytest
import torch

import moe_swiglu_epilogue_gb300 as M


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(M, "_lib", None)
    monkeypatch.setattr(M, "library_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(ImportError, match="no fallback"):
        M.load_library()


@pytest.mark.parametrize("call", [
    lambda: M.moe_nvfp4_quantize(torch.zeros(4, 32, dtype=torch.bfloat16)),
    lambda: M.moe_nvfp4_quantize_scaled(torch.zeros(4, 32, dtype=torch.bfloat16), 1.5),
    lambda: M.moe_swiglu_nvfp4_quantize(torch.zeros(4, 64, dtype=torch.bfloat16), 7.0),
    lambda: M.moe_swiglu_nvfp4_quantize_ex(torch.zeros(4, 64, dtype=torch.bfloat16), 7.0, global_scale=1.25),
    lambda: M.moe_swiglu_bf16(torch.zeros(4, 64, dtype=torch.bfloat16), 7.0),
    lambda: M.moe_nvfp4_dequantize(torch.zeros(4, 16, dtype=torch.uint8), torch.zeros(4, 2, dtype=torch.uint8)),
    lambda: M.moe_nvfp4_e4m3_codes(torch.zeros(8, dtype=torch.float32)),
], ids=["quantize", "quantize_scaled", "fused", "fused_ex", "compact_writer", "dequantize", "e4m3_codes"])
def test_cpu_tensors_are_refused(call):
    with pytest.raises((ValueError, TypeError), match="CUDA"):
        call()
