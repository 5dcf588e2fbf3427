"""The tensor wrappers refuse what the kernels cannot take, on any machine:
host tensors (the library has no CPU path) and types other than FP16 / BF16."""
import pytest
import torch

from polynomial_activation_gb300 import ops


@pytest.mark.parametrize("f", [ops.sigmoid, ops.tanh, ops.silu, ops.gelu,
                               lambda t: ops.softcap(t, 30.0),
                               lambda t: ops.swiglu_packed(t.view(8, 8)),
                               lambda t: ops.swiglu(t.view(8, 8), t.view(8, 8))])
def test_host_tensor_is_refused(f):
    x = torch.zeros(64, dtype=torch.float16)
    with pytest.raises(ValueError, match="no CPU path"):
        f(x)
    with pytest.raises(ValueError, match="no CPU path"):
        f(x.clone().requires_grad_(True))          # the recorded path refuses it too


def test_other_types_are_refused():
    with pytest.raises(TypeError):
        ops.silu(torch.zeros(64, dtype=torch.float32))
    with pytest.raises(TypeError):
        ops.swiglu(torch.zeros(4, 8, dtype=torch.float32), torch.zeros(4, 8, dtype=torch.float32))


def test_grad_decision():
    x = torch.zeros(4, dtype=torch.float16)
    assert not ops._grad(x)
    xr = x.clone().requires_grad_(True)
    assert ops._grad(xr) and ops._grad(x, xr)
    with torch.no_grad():
        assert not ops._grad(xr)
    with torch.inference_mode():
        assert not ops._grad(xr)


def test_packed_buffer_needs_an_even_last_dimension():
    with pytest.raises(ValueError, match="even"):
        ops.swiglu_packed(torch.zeros(4, 7, dtype=torch.float16))


def test_fused_base_detection():
    """ops.swiglu routes the two halves of one gate-up buffer in the graph to
    the fused-buffer path, and only those."""
    gu = torch.zeros(6, 10, dtype=torch.float16, requires_grad=True)
    g, u = gu.chunk(2, dim=-1)
    assert ops._fused_base(g, u) is gu
    assert ops._fused_base(u, g) is None                        # halves swapped
    root = torch.zeros(12, 10, requires_grad=True).half()       # a non-leaf buffer
    g, u = root.view(3, 4, 10).chunk(2, dim=-1)                 # through a reshape
    assert ops._fused_base(g, u) is root
    wide = torch.zeros(6, 15, requires_grad=True).half()
    assert ops._fused_base(wide[:, :5], wide[:, 5:10]) is None  # not the whole buffer
    other = torch.zeros(6, 5, dtype=torch.float16, requires_grad=True)
    assert ops._fused_base(gu[:, :5], other) is None            # u from another buffer
    plain = torch.zeros(6, 10, dtype=torch.float16)
    assert ops._fused_base(*plain.chunk(2, dim=-1)) is None     # no graph to route
    with torch.no_grad():
        g, u = gu.chunk(2, dim=-1)
    assert ops._fused_base(g, u) is None                        # views made without grad
    t = torch.zeros(10, 6, dtype=torch.float16, requires_grad=True).t()
    assert ops._fused_base(*t.chunk(2, dim=-1)) is None         # buffer not row-major


def test_unknown_swiglu_rule_is_refused():
    g = torch.zeros(8, 8, dtype=torch.bfloat16)
    for f in (lambda: ops.swiglu(g, g, rule=7), lambda: ops.swiglu_packed(g, rule=-1),
              lambda: ops.swiglu_ragged(g, g, torch.zeros(2, dtype=torch.int32), rule=2)):
        with pytest.raises(ValueError, match="rule"):
            f()
