"""The C-ABI library loads, exports every symbol include/moe.h declares, and
rejects bad configurations and arguments on the host (no GPU needed)."""
import ctypes as C
import os
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import int4_moe_expert_gb300 as m
    return m


def declared_functions():
    text = (ROOT / "include" / "moe.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_init", "moe_forward", "moe_forward_debug", "moe_forward_host", "moe_destroy",
              "moe_last_error", "moe_workspace_bytes", "moe_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(moe):
    L = C.CDLL(str(moe.library_path()))
    for name in declared_functions():
        assert hasattr(L, name), name


def test_config_struct_layout_matches_header(moe, tmp_path):
    """The ctypes structs have the header's size and field offsets (a C program
    compiled against include/moe.h prints them)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    fields = {"moe_config": moe.MoeConfig, "moe_weights": moe.MoeWeights}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe.h"', 'int main(void) {']
    for cname, py in fields.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run(["gcc", "-I", inc, str(src), "-o", str(exe)], check=True)
    out = dict(l.rsplit(" ", 1) for l in subprocess.run([str(exe)], check=True, capture_output=True,
                                                          text=True).stdout.splitlines())
    for cname, py in fields.items():
        assert int(out[f"{cname} size"]) == C.sizeof(py), cname
        for f, _ in py._fields_:
            assert int(out[f"{cname} {f}"]) == getattr(py, f).offset, (cname, f)


def test_workspace_bytes_validates_config(moe):
    good = moe.make_config(6144, 256, 8, 2048, 1, 2048, 2.5)
    assert moe.moe_workspace_bytes(good, 1) > 0
    assert moe.moe_workspace_bytes(good, 512) > moe.moe_workspace_bytes(good, 1)
    bad = [
        moe.make_config(6144, 256, 0, 2048, 1, 2048),        # K = 0
        moe.make_config(6144, 4, 8, 2048, 1, 2048),          # K > E
        moe.make_config(6144, 256, 33, 2048, 1, 2048),       # K > 32
        moe.make_config(6100, 256, 8, 2048, 1, 2048),        # H not a multiple of 32
        moe.make_config(6144, 256, 8, 2000, 1, 2048),        # I not a multiple of 32
        moe.make_config(6144, 256, 8, 2048, 1, 100),         # I_shared not a multiple of 32
        moe.make_config(6144, 256, 8, 2048, 2, 2048),        # two shared experts
        moe.make_config(6144, 256, 8, 2048, 1, 2048, n_group=3),           # E % n_group != 0
        moe.make_config(6144, 256, 8, 2048, 1, 2048, n_group=64, topk_group=4),   # n_group > 32
        moe.make_config(6144, 256, 8, 2048, 1, 2048, n_group=8, topk_group=0),
        moe.make_config(6144, 256, 8, 2048, 1, 2048, n_group=8, topk_group=9),
        moe.make_config(256, 16, 3, 128, 1, 128, n_group=8, topk_group=1),      # K > 1 group of 2
        moe.make_config(6144, 256, 8, 2048, 1, 2048, n_group=8, topk_group=4,
                        score_func=moe.MOE_SCORE_SOFTMAX),                    # groups need sigmoid
        moe.make_config(6144, 256, 8, 2048, 1, 2048, score_func=2),
        moe.make_config(6144, 256, 8, 2048, 1, 2048, expert_format=-1),
        moe.make_config(6144, 256, 8, 2048, 1, 2048, shared_format=3),
        moe.make_config(2048, 64, 8, 1056, expert_format=1),                  # int8: I % 128 != 0
        moe.make_config(2048, 64, 8, 1024, expert_format=1, cuda_cores=True),  # int8: tensor cores only
        moe.make_config(2048, 64, 8, 1056, expert_format=2),                  # group-64: I % 128 != 0
        moe.make_config(2048, 64, 8, 1024, expert_format=3),
        moe.make_config(6144, 2048, 8, 2048, 1, 2048),       # E > 1024
        moe.make_config(6144, 256, 8, 2048, 1, 2048, routed_scale=float("inf")),
    ]
    unknown_flag = moe.make_config(6144, 256, 8, 2048, 1, 2048)
    unknown_flag.flags = 16
    bad.append(unknown_flag)
    for cfg in bad:
        assert moe.moe_workspace_bytes(cfg, 1) == 0
    for cfg in (moe.make_config(6144, 256, 8, 2048, 1, 2048, 2.5, n_group=8, topk_group=4),
                moe.make_config(2048, 64, 8, 1024, score_func=moe.MOE_SCORE_SOFTMAX),
                moe.make_config(2048, 64, 8, 1024, norm_topk=0, score_func=moe.MOE_SCORE_SOFTMAX),
                moe.make_config(2048, 64, 8, 1024, expert_format=moe.MOE_FORMAT_INT8),
                moe.make_config(6144, 256, 8, 2048, 1, 2048, shared_format=moe.MOE_FORMAT_INT8),
                moe.make_config(2048, 256, 4, 512, 1, 512, expert_format=moe.MOE_FORMAT_G64,
                                shared_format=moe.MOE_FORMAT_G64)):
        assert moe.moe_workspace_bytes(cfg, 4) > 0
    # the trace flag is accepted and adds the trace buffer (1024 blocks x 64 x 8 B)
    traced = moe.make_config(6144, 256, 8, 2048, 1, 2048, 2.5, trace=True)
    assert moe.moe_workspace_bytes(traced, 1) >= moe.moe_workspace_bytes(good, 1) + 1024 * 64 * 8
    assert moe.moe_workspace_bytes(good, 0) == 0
    assert moe.moe_workspace_bytes(good, 1 << 20) == 0


def test_workspace_grows_linearly_in_max_tokens(moe):
    """The workspace is per-token buffers (h, down outputs, f16 activations, routing) plus
    the tiled router's partial logits, which are bounded in rows (split count x tokens):
    about 0.4 MB per token on the GLM layer from 64 tokens up, never a quadratic term.
    Handles for 256 tokens or more add the tcgen05 path's item-blocked f16 activations:
    128 rows of H + I values for each work item a call can have (T K / 128 full items, one
    partial item per expert, the shared expert's items)."""
    H, E, K, I = 6144, 256, 8, 2048
    glm = moe.make_config(H, E, K, I, 1, I, 2.5)
    sizes = {T: moe.moe_workspace_bytes(glm, T) for T in (64, 255, 256, 512, 4096, 16384)}

    def tc_blocks(T):
        items = T * K // 128 + min(E, T * K) + (T + 127) // 128 + 1
        return items * 128 * (H + I) * 2

    for T, b in sizes.items():
        extra = tc_blocks(T) if T >= 256 else 0
        assert 0 < (b - extra) / T < 420_000, (T, b, extra)
    assert sizes[255] + tc_blocks(256) - 2 * 256 * (K + 1) * I < sizes[256]
    assert sizes[512] < sizes[4096] < sizes[16384]


def test_null_arguments_are_errors_not_crashes(moe):
    L = moe.lib()
    cfg = moe.make_config(256, 16, 2, 128, 1, 128, 2.5)
    h = C.c_void_p(123)
    assert L.moe_init(C.byref(cfg), None, 1, C.byref(h)) == moe.MOE_ERR_INVALID
    assert h.value is None
    assert "weights" in moe.moe_last_error()
    assert L.moe_init(None, None, 1, C.byref(h)) == moe.MOE_ERR_INVALID
    assert L.moe_forward(None, None, 1, None, None) == moe.MOE_ERR_INVALID
    assert L.moe_forward_host(None, None, 1, None, None) == moe.MOE_ERR_INVALID
    assert L.moe_destroy(None) == moe.MOE_OK
    cfg_bad = moe.make_config(256, 16, 2, 128, 1, 128, n_group=3)
    assert L.moe_init(C.byref(cfg_bad), None, 1, C.byref(h)) == moe.MOE_ERR_INVALID
    assert "n_group" in moe.moe_last_error()
    with pytest.raises(moe.MoeError):
        moe.moe_forward(0, None, 1, None, stream=0)


def test_abi_version(moe):
    assert moe.moe_abi_version() == 4


def test_product_path_does_not_reference_the_oracle():
    pkg = ROOT / "int4_moe_expert_gb300"
    for f in list(pkg.rglob("*.py")) + list(pkg.rglob("*.cu")) + list(pkg.rglob("*.h")):
        text = f.read_text()
        assert "oracle" not in text.lower(), f
