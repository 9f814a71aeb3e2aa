"""CPU-only checks of the C ABI: the library loads, exports every symbol that
include/moe.h declares, and rejects bad arguments synchronously (no GPU call
is reached on those paths)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from moe_expert_routing_route_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build_library()
    return binding.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_route_topk", "moe_init_routing", "moe_grouped_ffn", "moe_finalize_routing",
              "moe_layer_forward"):
        assert n in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported by libmoe.so"
        assert name in binding.SIGNATURES, f"{name} has no binding signature"


def test_status_strings(lib):
    assert lib.moe_abi_version() == 2
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(4) == b"MOE_ERR_DEVICE"


def test_invalid_arguments_return_synchronously(lib):
    P = ctypes.c_void_p
    fake = P(256)  # never dereferenced: validation fails first
    # k > E
    assert lib.moe_route_topk(fake, None, 4, 2, 3, 1, fake, fake, None) == binding.MOE_ERR_INVALID_ARG
    # E > 1024
    assert lib.moe_route_topk(fake, None, 4, 2000, 3, 1, fake, fake, None) == binding.MOE_ERR_INVALID_ARG
    # null outputs
    assert lib.moe_route_topk(fake, None, 4, 8, 2, 1, None, fake, None) == binding.MOE_ERR_INVALID_ARG
    # H not a multiple of 8
    assert lib.moe_gate_logits(fake, fake, binding.MOE_BF16, 4, 12, 8, fake, None) == binding.MOE_ERR_UNSUPPORTED
    # misaligned pointer
    assert lib.moe_gate_logits(P(258), fake, binding.MOE_BF16, 4, 16, 8, fake, None) == binding.MOE_ERR_UNSUPPORTED
    # workspace too small
    assert lib.moe_init_routing(fake, 1, fake, 4, 16, 8, 2, fake, fake, fake, fake, fake, 8, None) == \
        binding.MOE_ERR_INVALID_ARG
    # grouped FFN without offsets needs E == 1
    assert lib.moe_grouped_ffn(fake, 1, None, 4, 16, 16, 16, fake, fake, fake, fake, 1 << 20, None) == \
        binding.MOE_ERR_INVALID_ARG
    # T == 0 is a no-op
    assert lib.moe_route_topk(None, None, 0, 8, 2, 1, None, None, None) == binding.MOE_OK


def test_layer_workspace_layout(lib):
    d = binding.LayerDesc(4096, 7168, 256, 8, 2048, 1, binding.MOE_BF16, 1, 256, 0, 256, 256, 256, 256)
    total = lib.moe_layer_workspace_bytes(ctypes.byref(d))
    R = 4096 * 8
    assert total > 2 * R * 7168 * 2  # expanded_x and y_routed
    prev_end = binding.MOE_WS_HEADER_BYTES
    for f, name in enumerate(binding.WS_FIELDS):
        off, nb = ctypes.c_size_t(), ctypes.c_size_t()
        assert lib.moe_layer_workspace_field(ctypes.byref(d), f, ctypes.byref(off), ctypes.byref(nb)) == 0
        assert off.value % 256 == 0 and off.value >= prev_end
        prev_end = off.value + nb.value
    assert prev_end <= total
    sizes = {}
    for name in ("expanded_x", "y_routed", "logits"):
        off, nb = ctypes.c_size_t(), ctypes.c_size_t()
        lib.moe_layer_workspace_field(ctypes.byref(d), binding.WS_FIELDS.index(name), ctypes.byref(off),
                                      ctypes.byref(nb))
        sizes[name] = nb.value
    # the logits region has room for the gate GEMM's K slices (8 at most)
    assert sizes == {"expanded_x": R * 7168 * 2, "y_routed": R * 7168 * 2, "logits": 8 * 4096 * 256 * 4}


def test_packed_weight_size(lib):
    # I = 1408 = 11 * 128: no padding; I = 200 pads to 256 rows of gate and of up
    assert lib.moe_w13_packed_bytes(binding.MOE_BF16, 64, 2048, 1408) == 64 * 2 * 1408 * 2048 * 2
    assert lib.moe_w13_packed_bytes(binding.MOE_F32, 3, 16, 200) == 3 * 2 * 256 * 16 * 4


def test_stage_names(lib):
    assert binding.stage_names()[0] == "gate" and binding.stage_names()[-1] == "finalize"
