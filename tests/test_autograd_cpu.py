"""Host-side checks of the autograd entry point (no GPU needed)."""
import pytest
import torch

from vocab_selected_token_tile_gb300.autograd import selected_logprob


def test_rejects_cpu_or_non_bf16_logits_before_any_call():
    with pytest.raises(TypeError):
        selected_logprob(torch.zeros(4, 16, dtype=torch.bfloat16), torch.zeros(4, dtype=torch.int64))
    with pytest.raises(TypeError):
        selected_logprob(torch.zeros(4, 16, dtype=torch.float32), torch.zeros(4, dtype=torch.int64))


def test_lmhead_autograd_rejects_cpu_or_non_bf16_inputs_before_any_call():
    from vocab_selected_token_tile_gb300.autograd import lmhead_logprob
    with pytest.raises(TypeError):
        lmhead_logprob(torch.zeros(4, 64, dtype=torch.bfloat16), torch.zeros(16, 64, dtype=torch.bfloat16),
                       torch.zeros(4, dtype=torch.int64))
    with pytest.raises(TypeError):
        lmhead_logprob(torch.zeros(4, 64, dtype=torch.float32), torch.zeros(16, 64, dtype=torch.float32),
                       torch.zeros(4, dtype=torch.int64))
