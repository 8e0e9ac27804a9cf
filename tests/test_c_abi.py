"""The boundary from plain C: moe_ffn.h compiles as C99 and C programs link
libmoe_ffn.so with no PyTorch in the process.

The first program checks what the host decides before any launch (no GPU
needed): workspace sizes, the unsupported-dims and argument errors, and the
status strings.  The second (GPU) allocates device memory with cudaMalloc,
copies seeded inputs in, runs moe_infer and moe_permute on the default stream
and writes the results back for comparison with the binding and the oracle."""

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


GPU_PROGRAM = r"""
/* moe_infer and moe_permute from plain C: device memory from cudaMalloc, the default stream. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime_api.h>
#include "moe_ffn.h"

static const char *dir;

static void *upload(const char *name, size_t bytes)
{
    char path[4096];
    void *h, *d = NULL;
    FILE *f;
    snprintf(path, sizeof path, "%s/%s", dir, name);
    f = fopen(path, "rb");
    if (!f) return NULL;
    h = malloc(bytes);
    if (!h || fread(h, 1, bytes, f) != bytes) { fclose(f); free(h); return NULL; }
    fclose(f);
    if (cudaMalloc(&d, bytes) != cudaSuccess || cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) d = NULL;
    free(h);
    return d;
}

static int download(const char *name, const void *d, size_t bytes)
{
    char path[4096];
    void *h = malloc(bytes);
    FILE *f;
    int ok;
    snprintf(path, sizeof path, "%s/%s", dir, name);
    if (!h || cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) { free(h); return 0; }
    f = fopen(path, "wb");
    ok = f && fwrite(h, 1, bytes, f) == bytes;
    if (f) fclose(f);
    free(h);
    return ok;
}

int main(int argc, char **argv)
{
    moe_dims dm;
    moe_weights w;
    size_t n, d, f, E, k, ws_bytes, pws_bytes;
    void *x, *ids, *wt, *y = NULL, *ws = NULL, *pws = NULL, *counts = NULL, *offsets = NULL, *sp = NULL;
    moe_status st;
    if (argc != 7) return 2;
    dir = argv[1];
    n = (size_t)atol(argv[2]);
    dm.d = atoi(argv[3]); dm.d_ff = atoi(argv[4]); dm.num_experts = atoi(argv[5]); dm.top_k = atoi(argv[6]);
    dm.act_scheme = MOE_ACT_EXACT;
    d = (size_t)dm.d; f = (size_t)dm.d_ff; E = (size_t)dm.num_experts; k = (size_t)dm.top_k;
    x = upload("x.bin", n * d * 2);
    ids = upload("ids.bin", n * k * 4);
    wt = upload("w.bin", n * k * 4);
    memset(&w, 0, sizeof w);
    w.w_gate = upload("w_gate.bin", E * f * d);
    w.w_up = upload("w_up.bin", E * f * d);
    w.w_down = upload("w_down.bin", E * d * f);
    w.s_gate = upload("s_gate.bin", E * (f / 128) * (d / 128) * 4);
    w.s_up = upload("s_up.bin", E * (f / 128) * (d / 128) * 4);
    w.s_down = upload("s_down.bin", E * (d / 128) * (f / 128) * 4);
    w.layout = MOE_LAYOUT_ROW_MAJOR;
    if (!x || !ids || !wt || !w.w_gate || !w.w_up || !w.w_down || !w.s_gate || !w.s_up || !w.s_down) return 3;
    ws_bytes = moe_workspace_size(&dm, (int64_t)n, 0);
    pws_bytes = moe_permute_workspace_size(&dm, (int64_t)n);
    if (!ws_bytes || !pws_bytes) return 4;
    if (cudaMalloc(&y, n * d * 2) != cudaSuccess || cudaMalloc(&ws, ws_bytes) != cudaSuccess ||
        cudaMalloc(&pws, pws_bytes) != cudaSuccess || cudaMalloc(&counts, E * 4) != cudaSuccess ||
        cudaMalloc(&offsets, (E + 1) * 4) != cudaSuccess || cudaMalloc(&sp, n * k * 4) != cudaSuccess)
        return 5;
    st = moe_infer(&dm, (int64_t)n, x, (const int32_t *)ids, (const float *)wt, &w, y, 0, ws, ws_bytes, NULL, NULL);
    if (st != MOE_OK) { fprintf(stderr, "moe_infer: %s\n", moe_status_string(st)); return 6; }
    st = moe_get_error(ws, NULL);
    if (st != MOE_OK) { fprintf(stderr, "device: %s\n", moe_status_string(st)); return 7; }
    st = moe_permute(&dm, (int64_t)n, (const int32_t *)ids, (int32_t *)counts, (int32_t *)offsets, (int32_t *)sp,
                     NULL, 0, pws, pws_bytes, NULL);
    if (st != MOE_OK || moe_get_error(pws, NULL) != MOE_OK) return 8;
    if (cudaDeviceSynchronize() != cudaSuccess) return 9;
    if (!download("y.bin", y, n * d * 2) || !download("counts.bin", counts, E * 4) ||
        !download("sorted_pos.bin", sp, n * k * 4))
        return 10;
    printf("ok\n");
    return 0;
}
"""


def _cudart_dir():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if not cand:
            continue
        for sub in ["lib64"] + [os.path.join("targets", t, "lib") for t in ("sbsa-linux", "x86_64-linux")]:
            p = os.path.join(cand, sub)
            if os.path.exists(os.path.join(p, "libcudart.so")):
                return p
    return None


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


@pytest.mark.gpu
@pytest.mark.parametrize("wl", ["tiny",                                           # wide tiles
                                ("c16s", 37, 512, 256, 5, 3, 44)])                # 16-token tiles
def test_c_program_runs_the_forward_on_the_gpu(wl):
    """The forward driven from C99 alone (cudaMalloc, cudaMemcpy, the default stream): its output is
    byte-identical to the binding's on the same inputs and within the tolerance of the oracle, and its
    routing plan equals the oracle's stable sort."""
    import numpy as np
    import torch
    import oracle
    from mixture_experts_ffn_infer_gb300 import synthetic as syn
    if shutil.which("gcc") is None or _cuda_include() is None or _cudart_dir() is None:
        pytest.skip("needs gcc, the CUDA headers and libcudart")
    w = syn.WORKLOADS[wl] if isinstance(wl, str) else syn.Workload(wl[0], *wl[1:6], seed=wl[6])
    inp = syn.make_inputs(w)
    n, d, dff, E, k = w.n_tokens, w.d, w.d_ff, w.num_experts, w.top_k
    with tempfile.TemporaryDirectory() as tmp:
        def put(name, t):
            t.contiguous().view(torch.uint8).numpy().tofile(os.path.join(tmp, name))
        put("x.bin", inp.x.view(torch.int16))
        put("ids.bin", inp.topk_ids.to(torch.int32))
        put("w.bin", inp.topk_weight.to(torch.float32))
        b = inp.bank
        for name in ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down"):
            put(name + ".bin", getattr(b, name))
        src, exe = os.path.join(tmp, "fwd.c"), os.path.join(tmp, "fwd")
        open(src, "w").write(GPU_PROGRAM)
        libdir = os.path.dirname(mx.LIB_PATH)
        subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                               "-I", _cuda_include(), src, "-o", exe, mx.LIB_PATH, "-L", _cudart_dir(), "-lcudart",
                               "-Wl,-rpath," + libdir + ":" + _cudart_dir()])
        out = subprocess.run([exe, tmp, str(n), str(d), str(dff), str(E), str(k)], capture_output=True, text=True,
                             timeout=120)
        assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
        y = torch.from_numpy(np.fromfile(os.path.join(tmp, "y.bin"), dtype=np.int16)).view(torch.bfloat16)
        y = y.reshape(n, d)
        counts = np.fromfile(os.path.join(tmp, "counts.bin"), dtype=np.int32)
        sp = np.fromfile(os.path.join(tmp, "sorted_pos.bin"), dtype=np.int32)
    bank_d = syn.ExpertBank(*(t.cuda() for t in (b.w_gate, b.w_up, b.w_down, b.s_gate, b.s_up, b.s_down)))
    y_py = mx.infer(inp.x.cuda(), inp.topk_ids.cuda(), inp.topk_weight.cuda(), bank_d).cpu()
    assert torch.equal(y.view(torch.int16), y_py.view(torch.int16))
    rep = oracle.parity_report(y, oracle.moe_infer(inp.x, inp.topk_ids, inp.topk_weight, b), True)
    assert rep["ok"], rep
    ref = oracle.permute(inp.topk_ids, E)
    assert np.array_equal(counts, np.asarray(ref[0])) and np.array_equal(sp, np.asarray(ref[2]))
