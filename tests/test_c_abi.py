"""The boundary from plain C: moe_ffn.h compiles as C99 and a C program links
libmoe_ffn.so and calls its host-side entry points (no GPU needed).

The program checks what the host decides before any launch: workspace sizes,
the unsupported-dims and argument errors, and the status strings."""

import os
import shutil
import subprocess
import tempfile

import pytest

import mixture_experts_ffn_infer_gb300 as mx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "moe_ffn.h"

int main(void)
{
    moe_dims k2 = {7168, 2048, 384, 8, MOE_ACT_EXACT};
    moe_dims fp8 = {7168, 2048, 384, 8, MOE_ACT_FP8_DYNAMIC};
    moe_dims bad_d = {7168 + 64, 2048, 384, 8, MOE_ACT_EXACT};
    moe_dims bad_act = {7168, 2048, 384, 8, 7};
    moe_dims mlp = {1024, 256, 1, 1, MOE_ACT_EXACT};
    moe_weights w;
    memset(&w, 0, sizeof w);
    size_t a = moe_workspace_size(&k2, 16, 0), b = moe_workspace_size(&k2, 4096, 2048);
    if (a == 0 || b <= a) return 1;
    if (moe_workspace_size(&fp8, 4096, 2048) != b) return 2;
    if (moe_workspace_size(&bad_d, 16, 0) != 0 || moe_workspace_size(&bad_act, 16, 0) != 0) return 3;
    if (moe_permute_workspace_size(&k2, 16) == 0 || moe_permute_workspace_size(&k2, 16) >= a) return 4;
    if (moe_tiled_bytes(0, 384, 7168, 2048) != (size_t)2 * 384 * 2048 * 7168) return 5;
    /* host-detected errors come back before anything is launched */
    if (moe_infer(&k2, 8, NULL, NULL, NULL, &w, NULL, 0, NULL, 0, NULL, NULL) != MOE_ERR_WORKSPACE) return 6;
    if (moe_infer(&bad_d, 8, NULL, NULL, NULL, &w, NULL, 0, NULL, 0, NULL, NULL) != MOE_ERR_UNSUPPORTED) return 7;
    if (moe_mlp_forward(&k2, 8, NULL, &w, NULL, 0, NULL, 0, NULL) != MOE_ERR_UNSUPPORTED) return 8;
    if (moe_mlp_forward(&mlp, 0, NULL, &w, NULL, 0, NULL, 0, NULL) != MOE_ERR_WORKSPACE) return 9;
    if (moe_combine(&k2, 0, NULL, NULL, NULL, NULL, 0, NULL) != MOE_OK) return 10;
    if (moe_get_error(NULL, NULL) != MOE_ERR_INVALID_ARG) return 11;
    if (strcmp(moe_status_string(MOE_ERR_ROUTING), "MOE_ERR_ROUTING") != 0) return 12;
    printf("ok %zu %zu\n", a, b);
    return 0;
}
"""


def _cuda_include():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return os.path.join(cand, "include")
    return None


@pytest.mark.skipif(shutil.which("gcc") is None or _cuda_include() is None, reason="needs gcc and the CUDA headers")
def test_c_program_uses_the_boundary():
    lib = mx.LIB_PATH
    if not os.path.exists(lib):
        pytest.skip("library not built")
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "abi.c")
        exe = os.path.join(tmp, "abi")
        open(src, "w").write(PROGRAM)
        subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                               "-I", _cuda_include(), src, "-o", exe, lib,
                               "-Wl,-rpath," + os.path.dirname(lib)])
        out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
        assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
        assert out.stdout.startswith("ok ")
