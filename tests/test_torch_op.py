"""The torch.library custom op around the C ABI: its fake implementation on
the CPU, and on the GPU the same results eagerly and under torch.compile."""
import pytest
import torch

from head_attention_forward_fmha_gb300 import inputs, torch_op


def test_op_is_registered_with_fake_shapes():
    from torch._subclasses.fake_tensor import FakeTensorMode
    with FakeTensorMode():
        q = torch.empty((2, 8, 3, 128), dtype=torch.bfloat16)
        k = torch.empty((2, 2, 70, 128), dtype=torch.bfloat16)
        o, lse = torch.ops.fmha_gb300.fwd(q, k, k, 0.1, 0, True)
    assert tuple(o.shape) == (2, 8, 3, 128) and o.dtype == torch.bfloat16
    assert tuple(lse.shape) == (2, 8, 3) and lse.dtype == torch.float32


@pytest.mark.gpu
def test_op_eager_and_compiled_match():
    from check_utils import compare, oracle_full
    w = inputs.Workload("op", 2, 16, 2, 4, 300, 128, window=100, causal=True)
    q, k, v = inputs.make_inputs(w, seed=41)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()

    def f(a, b, c):
        o, lse = torch_op.attention(a, b, c, w.scale, w.window, w.causal)
        return o.float() * 2.0, lse

    o1, l1 = f(qd, kd, vd)
    o2, l2 = torch.compile(f, backend="aot_eager", fullgraph=True)(qd, kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o_ref, lse_ref = oracle_full(w, q, k, v)
    compare(o1 / 2.0, l1, o_ref, lse_ref, "custom op")


def test_op_fake_shapes_with_sink():
    from torch._subclasses.fake_tensor import FakeTensorMode
    with FakeTensorMode():
        q = torch.empty((1, 4, 1, 64), dtype=torch.bfloat16)
        k = torch.empty((1, 1, 9, 64), dtype=torch.bfloat16)
        o, lse = torch.ops.fmha_gb300.fwd(q, k, k, 0.125, 0, False, torch.empty(4))
    assert tuple(o.shape) == (1, 4, 1, 64) and tuple(lse.shape) == (1, 4, 1)


@pytest.mark.gpu
def test_op_with_sink_matches_oracle():
    import oracle
    from check_utils import compare, to_np_bits
    w = inputs.Workload("op_sink", 1, 8, 2, 2, 200, 128, causal=True)
    q, k, v = inputs.make_inputs(w, seed=42)
    sink = torch.linspace(-2.0, 3.0, w.n_h, dtype=torch.float64)
    o, lse = torch_op.attention(q.cuda(), k.cuda(), v.cuda(), w.scale, w.window, w.causal,
                                sink=sink.float().cuda())
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(to_np_bits(q), to_np_bits(k), to_np_bits(v), w.scale, w.window, w.causal,
                                      sink=sink.float().double().numpy())
    compare(o, lse, o_ref, lse_ref, "custom op with sink")
