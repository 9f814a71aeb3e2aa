"""CPU-only: the ctypes binding agrees with include/moe.h.

The binding restates the header's struct layout, constants and function
signatures by hand; a drift between the two would pass wrong arguments to the
library without any error.  A small C program compiled against the header with
the host compiler prints the struct's size and field offsets and every constant
the binding mirrors, and the declarations are parsed for their parameter
kinds, so that each side is checked against the header itself."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from moe_expert_routing_route_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def _header_without_comments() -> str:
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    return re.sub(r"//[^\n]*", " ", src)


def _declarations() -> dict:
    """name -> (return type text, [parameter type texts]) for every moe_* function."""
    src = _header_without_comments()
    out = {}
    for m in re.finditer(r"([A-Za-z_][\w\s\*]*?)\b(moe_[a-z0-9_]+)\s*\(([^;{}]*?)\)\s*;", src):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        if name in out:
            continue
        if params in ("", "void"):
            plist = []
        else:
            plist = [p.strip() for p in params.split(",")]
        # the type of a parameter is its text without the trailing name
        types = [re.sub(r"\b\w+\s*$", "", p).strip() if re.search(r"[\w\*]\s+\**\w+$", p) else p for p in plist]
        out[name] = (ret.split()[-1] if ret else ret, types, ret)
    return out


def _kind_of_c(t: str) -> str:
    t = " ".join(t.replace("const", " ").split())
    if "*" in t or t == "moe_stream_t":
        return "ptr"
    if t in ("size_t", "uint64_t", "unsigned long long"):
        return "u64"  # ctypes names one 8-byte unsigned type for all three on a 64-bit host
    if t == "int64_t":
        return "i64"
    if t in ("int", "int32_t", "moe_status_t", "moe_dtype_t", "moe_ws_field", "moe_ws_field_ep", "uint32_t"):
        return "int"
    raise AssertionError(f"unclassified C type {t!r}")


def _kind_of_ctypes(t) -> str:
    if t in (ctypes.c_void_p, ctypes.c_char_p) or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "ptr"
    if t in (ctypes.c_size_t, ctypes.c_uint64):
        return "u64"
    if t is ctypes.c_int64:
        return "i64"
    if t in (ctypes.c_int, ctypes.c_int32, ctypes.c_uint32):
        return "int"
    raise AssertionError(f"unclassified ctypes type {t!r}")


def test_every_signature_matches_the_header():
    decls = _declarations()
    assert len(decls) >= 30
    for name, (restype, argtypes) in binding.SIGNATURES.items():
        assert name in decls, f"{name} bound but not declared"
        _, ctypes_params, ret_text = decls[name]
        want = [_kind_of_c(t) for t in ctypes_params]
        got = [_kind_of_ctypes(t) for t in argtypes]
        assert got == want, f"{name}: binding {got} against header {want}"
        ret_kind = "ptr" if "*" in ret_text else _kind_of_c(ret_text.split()[-1])
        assert _kind_of_ctypes(restype) == ret_kind, f"{name}: return type"


def test_layer_desc_struct_and_constants_match_the_header(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    fields = [f for f, _ in binding.LayerDesc._fields_]
    consts = ["MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_UNSUPPORTED", "MOE_ERR_CUDA", "MOE_ERR_DEVICE", "MOE_F32",
              "MOE_BF16", "MOE_DEVERR_BAD_EXPERT_ID", "MOE_DEVERR_BAD_ROW_INDEX", "MOE_DEVERR_BAD_OFFSETS",
              "MOE_DEVERR_TIMEOUT", "MOE_WS_HEADER_BYTES", "MOE_NUM_STAGES", "MOE_WEIGHTS_NATIVE", "MOE_WEIGHTS_FP8",
              "MOE_WEIGHTS_FP8_POW2", "MOE_LAYOUT_ROWS", "MOE_LAYOUT_TILED", "MOE_WS_NUM_FIELDS",
              "MOE_WS_EP_NUM_FIELDS"]
    ws = ["MOE_WS_" + n.upper() for n in binding.WS_FIELDS]
    ws_ep = ["MOE_WS_EP_" + n.upper() for n in binding.WS_FIELDS_EP]
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe.h"', "int main(void) {",
             'printf("sizeof %zu\\n", sizeof(moe_layer_desc));']
    lines += [f'printf("off {f} %zu\\n", offsetof(moe_layer_desc, {f}));' for f in fields]
    lines += [f'printf("const {c} %lld\\n", (long long)({c}));' for c in consts + ws + ws_ep]
    lines += ["return 0; }"]
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "probe"
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                        str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60, check=True).stdout.split("\n")
    vals = {}
    for line in out:
        parts = line.split()
        if len(parts) == 2:
            vals[parts[0]] = int(parts[1])
        elif len(parts) == 3:
            vals[(parts[0], parts[1])] = int(parts[2])
    # the struct: same size, every field at the same offset, no field the binding leaves out
    assert vals["sizeof"] == ctypes.sizeof(binding.LayerDesc)
    for f in fields:
        assert vals[("off", f)] == getattr(binding.LayerDesc, f).offset, f
    # constants mirrored in the binding
    mirrored = {"MOE_OK": binding.MOE_OK, "MOE_ERR_INVALID_ARG": binding.MOE_ERR_INVALID_ARG,
                "MOE_ERR_UNSUPPORTED": binding.MOE_ERR_UNSUPPORTED, "MOE_ERR_CUDA": binding.MOE_ERR_CUDA,
                "MOE_ERR_DEVICE": binding.MOE_ERR_DEVICE, "MOE_F32": binding.MOE_F32, "MOE_BF16": binding.MOE_BF16,
                "MOE_DEVERR_BAD_EXPERT_ID": binding.MOE_DEVERR_BAD_EXPERT_ID,
                "MOE_DEVERR_BAD_ROW_INDEX": binding.MOE_DEVERR_BAD_ROW_INDEX,
                "MOE_DEVERR_BAD_OFFSETS": binding.MOE_DEVERR_BAD_OFFSETS,
                "MOE_DEVERR_TIMEOUT": binding.MOE_DEVERR_TIMEOUT, "MOE_WS_HEADER_BYTES": binding.MOE_WS_HEADER_BYTES,
                "MOE_NUM_STAGES": binding.MOE_NUM_STAGES, "MOE_WEIGHTS_NATIVE": binding.MOE_WEIGHTS_NATIVE,
                "MOE_WEIGHTS_FP8": binding.MOE_WEIGHTS_FP8, "MOE_WEIGHTS_FP8_POW2": binding.MOE_WEIGHTS_FP8_POW2,
                "MOE_LAYOUT_ROWS": binding.MOE_LAYOUT_ROWS, "MOE_LAYOUT_TILED": binding.MOE_LAYOUT_TILED,
                "MOE_WS_NUM_FIELDS": len(binding.WS_FIELDS), "MOE_WS_EP_NUM_FIELDS": len(binding.WS_FIELDS_EP)}
    for c, v in mirrored.items():
        assert vals[("const", c)] == v, c
    # workspace field names in enum order
    for i, c in enumerate(ws):
        assert vals[("const", c)] == i, c
    for i, c in enumerate(ws_ep):
        assert vals[("const", c)] == i, c
