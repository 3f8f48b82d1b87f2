"""MoeOp's argument checks, on the host (no GPU): a bad configuration is
refused when the op is made, before anything is enqueued."""
import pytest

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("kw,msg", [
    (dict(num_experts=0), "num_experts"),
    (dict(num_experts=1025), "num_experts"),
    (dict(num_experts=64, group_size=7), "divide"),
    (dict(num_experts=64, capacity=-1), ">= 0"),
    (dict(num_experts=64, quant_block=100), "power of two"),
    (dict(num_experts=64, quant_block=512), "power of two"),
    (dict(num_experts=64, quant_block=128, group_size=8), "dedup"),
    (dict(num_experts=64, out_dtype=torch.float16), "out_dtype"),
])
def test_bad_configurations_are_refused(kw, msg):
    import combine_moe_plan_02_gb300 as moe
    with pytest.raises(ValueError, match=msg):
        moe.MoeOp(**kw)


def test_modes_are_accepted():
    import combine_moe_plan_02_gb300 as moe
    for kw in (dict(), dict(capacity=640), dict(group_size=8), dict(quant_block=128),
               dict(capacity=100, group_size=8), dict(weighted=False, fold=False),
               dict(out_dtype=torch.float32)):
        op = moe.MoeOp(64, **kw)
        assert op.E == 64


def test_dispatch_checks_its_arguments_before_any_call():
    import combine_moe_plan_02_gb300 as moe
    op = moe.MoeOp(64)
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    idx = torch.zeros(4, 8, dtype=torch.int32)
    with pytest.raises(TypeError, match="topk_w"):
        op.dispatch(x, torch.zeros(4, 8, dtype=torch.float64), idx)
    with pytest.raises(TypeError, match="topk_idx"):
        op.dispatch(x, torch.zeros(4, 8), torch.zeros(4, 8, dtype=torch.float32))
    with pytest.raises(ValueError, match="x_scales"):
        moe.MoeOp(64, quant_block=128).dispatch(x, torch.zeros(4, 8), idx,
                                                x_scales=torch.zeros(4, 1))
