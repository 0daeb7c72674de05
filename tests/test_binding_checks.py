"""The binding's argument checks, on the CPU: the C ABI receives bare
pointers and cannot check buffer sizes, so the binding must refuse a wrongly
sized, typed, strided or placed tensor before any C call is made."""
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr

T, H, K, R = 4, 64, 8, 32


def _args():
    return dict(expert_out=torch.zeros((R, H), dtype=torch.bfloat16),
                permuted_row_of=torch.zeros((T, K), dtype=torch.int32),
                topk_weights=torch.zeros((T, K), dtype=torch.float32),
                residual_in=torch.zeros((T, H), dtype=torch.float32),
                residual_out=torch.zeros((T, H), dtype=torch.float32),
                gamma=torch.zeros((H,), dtype=torch.bfloat16), eps=1e-6,
                out=torch.zeros((T, H), dtype=torch.bfloat16))


@pytest.fixture
def no_c_call(monkeypatch):
    """Any attempt to reach the C library fails the test."""
    def refuse():
        raise AssertionError("the binding reached the C library")
    monkeypatch.setattr(mfr, "load_library", refuse)


@pytest.mark.parametrize("name,bad,match", [
    ("residual_out", torch.zeros((T - 1, H), dtype=torch.float32), "residual_out: expected"),
    ("residual_out", torch.zeros((T, H), dtype=torch.float64), "residual_out: expected"),
    ("out", torch.zeros((T, H), dtype=torch.float32), "out: expected"),
    ("gamma", torch.zeros((H + 8,), dtype=torch.bfloat16), "gamma: expected"),
    ("topk_weights", torch.zeros((T, K - 1), dtype=torch.float32), "topk_weights: expected"),
    ("residual_out", torch.zeros((H, T), dtype=torch.float32).t(), "residual_out must be contiguous"),
    ("residual_in", torch.zeros((T, 2 * H), dtype=torch.float32)[:, ::2], "residual_in must be contiguous"),
])
def test_run_noalloc_refuses_bad_tensors_without_a_call(no_c_call, name, bad, match):
    a = _args()
    a[name] = bad
    with pytest.raises(ValueError, match=match):
        mfr.run_noalloc(**a)


def test_run_noalloc_refuses_host_tensors_without_a_call(no_c_call):
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        mfr.run_noalloc(**_args())


def test_validate_fused_args_checks_every_tensor():
    a = _args()
    tensors = [a[n] for n in ("expert_out", "permuted_row_of", "topk_weights", "residual_in", "residual_out",
                              "gamma", "out")]
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        mfr.validate_fused_args(T, H, K, R, *tensors)
    for i in range(len(tensors)):
        bad = list(tensors)
        bad[i] = bad[i][:1] if bad[i].dim() == 1 else bad[i][:, :1]
        with pytest.raises(ValueError, match="expected"):
            mfr.validate_fused_args(T, H, K, R, *bad)
