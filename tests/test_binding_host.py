"""Host logic of the Python binding (no GPU): problem descriptors from tensor shapes and dtypes in
both layouts, rejection of host tensors before any call reaches the library, status codes raised
with the library's own status strings, and the forward workspace's size."""
import pytest
import torch

from relation_token_mixing_gb300 import binding as rb


def test_problem_for_both_layouts():
    t = torch.empty(2, 3, 5, 64, dtype=torch.bfloat16)
    p = rb.problem_for(t, 2.0, 0.5, True)
    assert (p.B, p.H, p.T, p.d_h, p.dtype, p.causal, p.layout) == (2, 3, 5, 64, rb.RELATION_BF16, 1,
                                                                   rb.RELATION_LAYOUT_BHTD)
    assert p.tau_S == 2.0 and p.lam == 0.5
    u = torch.empty(2, 5, 3, 60, dtype=torch.float32)  # [B, T, H, d]
    q = rb.problem_for(u, 1.0, 0.0, False, rb.RELATION_LAYOUT_BTHD)
    assert (q.B, q.H, q.T, q.d_h, q.dtype, q.causal, q.layout) == (2, 3, 5, 60, rb.RELATION_F32, 0,
                                                                   rb.RELATION_LAYOUT_BTHD)


def test_problem_for_rejects_what_the_library_has_no_kernel_for():
    with pytest.raises(ValueError):
        rb.problem_for(torch.empty(1, 1, 4, 64, dtype=torch.float16), 1.0, 0.5, True)
    with pytest.raises(ValueError):
        rb.problem_for(torch.empty(4, 64, dtype=torch.bfloat16), 1.0, 0.5, True)
    with pytest.raises(ValueError):
        rb.problem_for(torch.empty(1, 1, 4, 64, dtype=torch.bfloat16), 1.0, 0.5, True, layout=7)


def test_host_tensors_are_rejected_before_any_library_call():
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        rb.fwd(x, x, x, 1.0, 0.5, True)


def test_status_codes_raise_with_the_library_status_string():
    for code in range(1, 7):
        with pytest.raises(rb.RelationError) as e:
            rb._check(code, "relation_fwd")
        assert rb.relation_status_string(code) in str(e.value)
    rb._check(0, "relation_fwd")  # success raises nothing


def test_forward_workspace_only_for_rows_tma_cannot_address():
    p64 = rb.problem_for(torch.empty(1, 2, 100, 64, dtype=torch.bfloat16), 1.0, 0.5, True)
    assert rb.fwd_workspace(p64, "cpu") is None
    p60 = rb.problem_for(torch.empty(1, 2, 100, 60, dtype=torch.bfloat16), 1.0, 0.5, True)
    ws = rb.fwd_workspace(p60, "cpu")
    assert ws is not None and ws.numel() * ws.element_size() >= rb.relation_fwd_workspace_bytes(p60) > 0
