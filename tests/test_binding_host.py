"""The Python binding has no CPU path: every entry point refuses host tensors
with an error before any computation (no silent fallback), and the binding
refuses to import its functions when the library is missing."""
import pytest
import torch

from kv_cache_compression_attention_b300 import binding as B


def cpu(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


def i64(*shape):
    return torch.zeros(shape, dtype=torch.int64)


f32 = torch.float32
CALLS = {
    "kvc_score_attn": lambda: B.kvc_score_attn(cpu(1, 4, 8, 128), cpu(1, 2, 64, 128),
                                               cpu(1, 2, 64, dtype=f32), 0.1),
    "kvc_score_linear": lambda: B.kvc_score_linear(cpu(1, 64, 128), cpu(128, 2), None,
                                                   cpu(1, 2, 64, dtype=f32)),
    "kvc_score_mlp": lambda: B.kvc_score_mlp(cpu(1, 64, 128), cpu(128, 16), cpu(16, dtype=f32),
                                             cpu(16, 2), None, cpu(1, 2, 64, dtype=f32),
                                             workspace=cpu(1 << 10, dtype=torch.uint8)),
    "kvc_score_kvzip_plus": lambda: B.kvc_score_kvzip_plus(
        cpu(1, 4, 8, 128), cpu(1, 2, 64, 128), cpu(1, 2, 64, 128), cpu(4, 128, 128),
        cpu(1, 8, dtype=f32), cpu(1, 2, 64, dtype=f32), 0.1,
        workspace=cpu(1 << 10, dtype=torch.uint8)),
    "kvc_select": lambda: B.kvc_select(cpu(1, 2, 64, dtype=f32), "global", i32(2, 64), i32(2),
                                       i64(3), keep_ratio=0.5),
    "kvc_compact": lambda: B.kvc_compact(cpu(1, 2, 64, 128), cpu(1, 2, 64, 128), i32(2, 64),
                                         i32(2), i64(3), cpu(64, 128), cpu(64, 128), i64(2),
                                         i32(2)),
    "kvc_decode_attn": lambda: B.kvc_decode_attn(cpu(1, 4, 128), cpu(64, 128), cpu(64, 128),
                                                 i64(2), i32(2), cpu(1, 4, 128), max_len=64,
                                                 workspace=cpu(1 << 16, dtype=torch.uint8)),
    "kvc_quantize_rows": lambda: B.kvc_quantize_rows(cpu(64, 128), cpu(64, 128, dtype=torch.uint8),
                                                     cpu(64, 4, 2, dtype=torch.float16)),
    "kvc_decode_prune": lambda: B.kvc_decode_prune([cpu(64, 128), cpu(64, 128)],
                                                   cpu(64, dtype=f32), i64(2), i32(2),
                                                   cpu(2, dtype=f32), 0.5, 16),
    "kvc_gather_scores": lambda: B.kvc_gather_scores(cpu(1, 2, 64, dtype=f32), i32(2, 64),
                                                     i32(2), i64(2), cpu(64, dtype=f32)),
    "kvc_vector_residual": lambda: B.kvc_vector_residual(cpu(1, 2, 64, 128), cpu(1, 2, 64, 128),
                                                         cpu(2, 128, 128), i32(2, 64), i32(2),
                                                         cpu(1, 2, 64, dtype=f32)),
    "kvc_decode_attn_vector": lambda: B.kvc_decode_attn_vector(
        cpu(1, 4, 128), cpu(64, 128), cpu(64, 128), i64(2), i32(2), i64(2), i32(2),
        cpu(2, 128, 128), cpu(1, 4, 128), max_len=64,
        workspace=cpu(1 << 16, dtype=torch.uint8)),
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_entry_points_refuse_host_tensors(name):
    try:
        B.lib()
    except ImportError:
        pytest.skip("libkvc.so not built")
    with pytest.raises(ValueError, match="CUDA tensors"):
        CALLS[name]()


def test_missing_library_raises(tmp_path):
    with pytest.raises(ImportError):
        B.load(str(tmp_path / "libkvc.so"))
