"""The boundary from plain C (CPU only): a C99 program that includes only include/fcm.h and
links libfcm.so compiles with warnings as errors, runs without a GPU through the host-only
entry points (planner, tensor sizes, section IV cost models, FusePlanner over a chain), and
prints the same numbers the Python binding returns for the same calls."""
import os
import shutil
import subprocess

import pytest

import pointwise_conv_cnn_gb300 as fcm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include "fcm.h"

int main(void) {
    fcm_desc d = {0};
    fcm_plan_info info;
    size_t xb = 0, mb = 0, yb = 0;
    fcm_layer chain[2] = {{FCM_LAYER_DW, 4, 4, 32, 0, 3, 1, 1}, {FCM_LAYER_PW, 4, 4, 32, 32, 1, 1, 0}};
    fcm_layer_plan plans[2];
    long long total = 0;
    fcm_status st;

    d.n = 64; d.h = 56; d.w = 56; d.c = 128; d.k_out = 128;
    d.ksize = 3; d.stride = 1; d.pad = 1;
    d.conv1 = FCM_CONV1_DEPTHWISE; d.dtype = FCM_F16;
    d.act1 = FCM_ACT_RELU6; d.act2 = FCM_ACT_RELU6;
    st = fcm_plan_desc(&d, 152, 232448, &info);
    if (st != FCM_OK) { printf("plan failed: %s\n", fcm_last_error()); return 1; }
    printf("plan %d %d %d %d %d %d %d %lld %lld %lld\n", info.kernel, info.tile_h, info.tile_w,
           info.chunk_c, info.stages, info.ctas, info.smem_bytes, info.num_tiles,
           info.bytes_fused_min, info.bytes_unfused_min);
    if (fcm_tensor_bytes(&d, &xb, &mb, &yb) != FCM_OK) return 1;
    printf("bytes %zu %zu %zu\n", xb, mb, yb);

    d.c = 12; d.k_out = 12;                   /* 24-byte rows: refused, message set */
    st = fcm_plan_desc(&d, 152, 232448, &info);
    printf("misaligned %d %d\n", (int)st, fcm_last_error()[0] != '\0');

    printf("overlap %lld\n", fcm_model_overlap(56, 56, 28, 14, 3, 3, 1));
    st = fcm_fuse_plan(chain, 2, 1, 1, 2000000000LL, 2, plans, &total);
    printf("chain %d %lld %d %d %d\n", (int)st, total, plans[0].fuse_with_next, plans[0].module,
           plans[1].module);
    return 0;
}
"""


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fcm.load_library()
    d = tmp_path_factory.mktemp("c_consumer")
    src, exe = d / "consumer.c", d / "consumer"
    src.write_text(C_SOURCE)
    libdir = os.path.dirname(fcm.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", libdir, "-l:libfcm.so", "-Wl,-rpath," + libdir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return str(exe)


def test_c_program_matches_the_binding(program):
    r = subprocess.run([program], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    out = {ln.split()[0]: ln.split()[1:] for ln in r.stdout.splitlines()}

    d = fcm.make_desc(64, 56, 56, 128, 128, 3, 1, 1, conv1="dw", dtype="f16", act1="relu6",
                      act2="relu6")
    info = fcm.fcm_plan_desc(d, 152, 232448)
    want = [info[k] for k in ("kernel", "tile_h", "tile_w", "chunk_c", "stages", "ctas",
                              "smem_bytes", "num_tiles", "bytes_fused_min", "bytes_unfused_min")]
    assert list(map(int, out["plan"])) == want
    assert tuple(map(int, out["bytes"])) == fcm.fcm_tensor_bytes(d)
    assert out["misaligned"] == ["3", "1"]                     # FCM_ERR_ALIGNMENT + a message
    assert out["overlap"] == [str(fcm.fcm_model_overlap(56, 56, 28, 14, 3, 3, 1))]

    plans, total = fcm.fcm_fuse_plan([dict(kind="dw", h=4, w=4, c=32, ksize=3, stride=1, pad=1),
                                      dict(kind="pw", h=4, w=4, c=32, k_out=32)], 1, 1,
                                     2 * 10**9, 2)
    code = {name: k for k, name in fcm.MODULES.items()}
    assert out["chain"] == ["0", str(total), str(plans[0]["fuse_with_next"]),
                            str(code[plans[0]["module"]]), str(code[plans[1]["module"]])]
