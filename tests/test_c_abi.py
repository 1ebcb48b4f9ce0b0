"""The boundary from plain C (no GPU): a C11 program that includes only
include/moe.h, links libmoe.so and calls the host-side entry points.  It
checks that the header is valid C and that the library is usable without
Python.  The capacity check applies the capacity equation of "Mixture of
Experts" (module 17), 17.5, to the module's closing exercise: T=4096, k=8,
E=64 and capacity factor 1.25 give C=640;
rejected arguments must come back before any launch."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mixture_experts_layer_capacity_b300")
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "moe.h"

static moe_config cfg(int T, int D, int E, int F, int k, int S, int dtype, int mode, float gamma)
{
    moe_config c;
    memset(&c, 0, sizeof c);
    c.T = T; c.d_model = D; c.n_experts = E; c.d_expert = F; c.top_k = k; c.d_shared = S;
    c.dtype = dtype; c.gating_mode = mode; c.capacity_factor = gamma; c.aux_alpha = 0.01f;
    return c;
}

int main(void)
{
    moe_config ex = cfg(4096, 512, 64, 2048, 8, 0, MOE_DTYPE_BF16, MOE_GATE_SOFTMAX_ALL, 1.25f);
    moe_config sw = cfg(4096, 512, 8, 2048, 1, 0, MOE_DTYPE_BF16, MOE_GATE_SOFTMAX_ALL, 1.0f);
    moe_config bad = sw;
    size_t ws = 0;
    int32_t flags = -1;
    bad.n_experts = 16;
    bad.top_k = 9;
    printf("capacity_exercise %lld\n", (long long)moe_capacity(&ex));
    printf("capacity_switch %lld\n", (long long)moe_capacity(&sw));
    printf("workspace_status %d\n", (int)moe_workspace_size(&sw, &ws));
    printf("workspace_nonzero %d\n", ws > 0);
    printf("plan_status %d\n", (int)moe_launch_plan(&sw, &flags));
    printf("plan_router_fused %d\n", (flags & MOE_PLAN_ROUTER_FUSED) != 0);
    printf("plan_direct_y %d\n", (flags & MOE_PLAN_DIRECT_Y) != 0);
    printf("bad_k_status %d\n", (int)moe_workspace_size(&bad, &ws));
    printf("null_x_status %d\n",
           (int)moe_forward(&sw, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                            NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 0));
    printf("status_string %s\n", moe_status_string(MOE_ERR_WORKSPACE));
    {
        uint64_t words[8];
        size_t w8 = 0;
        moe_config wide = sw;
        wide.d_model = (1 << 20) + 64;
        printf("timeline_clear %d\n", (int)moe_timeline_clear());
        printf("timeline_read %d\n", (int)moe_timeline_read(words, 8));
        printf("w8a8_workspace_status %d\n", (int)moe_w8a8_workspace_size(&sw, &w8));
        printf("w8a8_workspace_covers %d\n", w8 >= ws);
        printf("wide_status %d\n", (int)moe_workspace_size(&wide, &ws));
        printf("capacity_huge %lld\n",
               (long long)moe_capacity(&(moe_config){4096, 512, 8, 2048, 2, 0, MOE_DTYPE_BF16,
                                                      MOE_GATE_SOFTMAX_ALL, 3.0e38f, 0.01f, 0}));
    }
    return 0;
}
"""


def _lib():
    path = os.path.join(PKG, "libmoe.so")
    if not os.path.exists(path):
        pytest.fail("libmoe.so is not built (run __graft_entry__.build())")
    return path


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_host_entry_points_from_c(tmp_path):
    _lib()
    src = tmp_path / "use_moe.c"
    exe = tmp_path / "use_moe"
    src.write_text(PROGRAM)
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), "-I", CUDA_INC, str(src),
           "-L", PKG, "-lmoe", f"-Wl,-rpath,{PKG}", "-o", str(exe)]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True,
                         timeout=120).stdout
    got = dict(line.split(" ", 1) for line in out.strip().splitlines())
    assert got["capacity_exercise"] == "640"
    assert got["capacity_switch"] == "512"
    assert got["workspace_status"] == "0" and got["workspace_nonzero"] == "1"
    assert got["plan_status"] == "0"
    assert got["plan_router_fused"] == "1" and got["plan_direct_y"] == "1"
    assert got["bad_k_status"] == "2"            # MOE_ERR_UNSUPPORTED: 8 < k <= E
    assert got["null_x_status"] == "1"           # MOE_ERR_INVALID_ARG
    assert "workspace" in got["status_string"].lower()
    # the timeline readers exist in every build and refuse outside theirs
    assert got["timeline_clear"] == "2" and got["timeline_read"] == "2"
    assert got["w8a8_workspace_status"] == "0" and got["w8a8_workspace_covers"] == "1"
    assert got["wide_status"] == "2"             # widths above 2^20
    assert got["capacity_huge"] == str(2**63 - 1)  # saturates, drops nothing
