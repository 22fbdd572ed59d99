"""The Python binding checks element types and shapes before it hands raw
pointers to the C ABI (a wrong dtype would otherwise be read as the wrong
element size); these checks run before any device work, so CPU tensors
exercise them."""
import pytest

torch = pytest.importorskip("torch")

import bit_expert_matvec_moe_b300 as M  # noqa: E402

D = M.Dims(hidden=256, inter=128, n_experts=16, top_k=4)


def _layer():
    # pointers given as integers are taken as they are (no tensor to check)
    return M.make_layer(D, 1 << 20, M.moe_packed_expert_bytes(D, 4), 2 << 20, shared=3 << 20)


@pytest.mark.parametrize("bad, msg", [
    (dict(h=torch.zeros((1, 256), dtype=torch.float16)), "h: expected dtype float32"),
    (dict(h=torch.zeros((1, 320), dtype=torch.float32)), "h: expected shape [B, 256]"),
    (dict(h=torch.zeros((256,), dtype=torch.float32)), "h: expected shape"),
    (dict(idx_out=torch.zeros((1, 4), dtype=torch.int64)), "idx_out: expected dtype int32"),
    (dict(w_out=torch.zeros((1, 3), dtype=torch.float32)), "w_out: expected at least 4 elements"),
    (dict(logit_offset=torch.zeros((1, 16), dtype=torch.float64)), "logit_offset: expected dtype float32"),
])
def test_layer_decode_argument_checks(bad, msg):
    args = dict(h=torch.zeros((1, 256), dtype=torch.float32))
    args.update(bad)
    h = args.pop("h")
    with pytest.raises(ValueError) as err:
        M.moe_layer_decode(_layer(), h, torch.zeros(16, dtype=torch.uint8), **args)
    assert msg in str(err.value)


def test_cpu_tensor_is_refused_after_type_checks():
    with pytest.raises(ValueError) as err:
        M.moe_layer_decode(_layer(), torch.zeros((1, 256), dtype=torch.float32), torch.zeros(16, dtype=torch.uint8))
    assert "expected a CUDA tensor" in str(err.value)


def test_router_and_pack_argument_checks():
    with pytest.raises(ValueError) as err:
        M.make_layer(D, 1 << 20, 64, torch.zeros((16, 256), dtype=torch.float32))
    assert "router: expected dtype" in str(err.value)
    with pytest.raises(ValueError) as err:
        M.make_layer(D, 1 << 20, 64, torch.zeros((8, 256), dtype=torch.int16))
    assert "router: expected at least 4096 elements" in str(err.value)
    codes = [torch.zeros((128, 128), dtype=torch.uint8)] * 3
    scales = [torch.zeros((128, 4), dtype=torch.float32)] * 3
    with pytest.raises(ValueError) as err:
        M.moe_pack_weights(D, 4, codes, scales, scales, 1 << 20)
    assert "scales: expected dtype" in str(err.value)
    with pytest.raises(ValueError) as err:
        M.moe_route(D, torch.zeros((2, 256), dtype=torch.float32), 1 << 20, torch.zeros((2, 4), dtype=torch.int32),
                    torch.zeros((2, 4), dtype=torch.float32), torch.zeros(16, dtype=torch.uint8),
                    logits_out=torch.zeros((2, 15), dtype=torch.float32))
    assert "logits_out: expected at least 32 elements" in str(err.value)


@pytest.mark.parametrize("bad, msg", [
    (dict(layers=[]), "no layers"),
    (dict(h=torch.zeros((1, 320), dtype=torch.float32)), "h must hold one token"),
    (dict(h=torch.zeros((2, 256), dtype=torch.float32)), "h must hold one token"),
    (dict(h=torch.zeros((1, 256), dtype=torch.float16)), "h: expected dtype float32"),
    (dict(idx_out=torch.zeros((2, 4), dtype=torch.int64)), "idx_out: expected dtype int32"),
    (dict(w_out=torch.zeros((2, 3), dtype=torch.float32)), "w_out: expected at least 8 elements"),
    (dict(logit_offset=torch.zeros((1, 16), dtype=torch.float32)), "logit_offset: expected at least 32 elements"),
])
def test_stack_decode_argument_checks(bad, msg):
    """moe_stack_decode: one token ([1, hidden] or [hidden]); per-layer rows of
    the offsets and outputs for every layer, checked before any device work."""
    args = dict(layers=[_layer(), _layer()], h=torch.zeros((1, 256), dtype=torch.float32))
    args.update(bad)
    layers, h = args.pop("layers"), args.pop("h")
    with pytest.raises(ValueError) as err:
        M.moe_stack_decode(layers, h, torch.zeros(16, dtype=torch.uint8), **args)
    assert msg in str(err.value)
