"""The header is plain C: a C99 program includes it, links libcacheblend.so and runs the host-side
checks (no GPU needed), and the binding's struct layouts match what a C compiler makes of the header."""

import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stddef.h>
#include <stdio.h>
#include <string.h>
#include "cacheblend.h"

int main(void) {
  cb_config c;
  cb_plan* plan = NULL;
  memset(&c, 0, sizeof(c));
  c.n_chunks = 2; c.chunk_len = 256; c.n_suffix = 32; c.hq = 4; c.hkv = 3; c.head_dim = 64;
  c.rope_theta = 1e4; c.rope_style = CB_ROPE_HALF; c.r1_pct = 15; c.r2_pct = 15;
  c.deviation = CB_DEV_V; c.filter = CB_FILTER_KEEP;
  /* hq not a multiple of hkv: rejected on the host, before any CUDA call */
  cb_status s = cb_plan_create(&c, &plan);
  printf("version %d\n", (int)cb_version());
  printf("plan_create %d %s %d\n", (int)s, plan == NULL ? "null" : "set", strstr(cb_last_error_string(), "multiple") != NULL);
  printf("blend_layer %d\n", (int)cb_blend_layer(NULL, 1, NULL, NULL));
  printf("config %zu %zu %zu %zu %zu\n", sizeof(cb_config), offsetof(cb_config, rope_theta),
         offsetof(cb_config, rope_style), offsetof(cb_config, deviation), offsetof(cb_config, filter));
  printf("layer_io %zu %zu %zu\n", sizeof(cb_layer_io), offsetof(cb_layer_io, cand), offsetof(cb_layer_io, out));
  return 0;
}
"""


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from rag_kv_cache_gb300.build import build

    lib = build()
    d = tmp_path_factory.mktemp("c_consumer")
    src = d / "consumer.c"
    src.write_text(C_SOURCE)
    exe = d / "consumer"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"), str(src),
                    lib, "-o", str(exe), f"-Wl,-rpath,{os.path.dirname(lib)}"], check=True, capture_output=True)
    return exe


def _run(exe):
    env = dict(os.environ)
    cuda_lib = "/usr/local/cuda/lib64"
    env["LD_LIBRARY_PATH"] = cuda_lib + (":" + env["LD_LIBRARY_PATH"] if env.get("LD_LIBRARY_PATH") else "")
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, env=env).stdout
    return dict((line.split()[0], line.split()[1:]) for line in out.strip().splitlines())


def test_c_program_compiles_links_and_runs_host_checks(consumer):
    r = _run(consumer)
    assert r["version"] == ["100"]
    assert r["plan_create"] == ["1", "null", "1"]  # CB_ERR_INVALID_ARG, no plan, message names the rule
    assert r["blend_layer"] == ["1"]


def test_binding_struct_layouts_match_the_c_compiler(consumer):
    from rag_kv_cache_gb300 import _lib

    r = _run(consumer)
    cfg = _lib.CbConfig
    assert [int(x) for x in r["config"]] == [ctypes.sizeof(cfg), cfg.rope_theta.offset, cfg.rope_style.offset,
                                             cfg.deviation.offset, cfg.filter.offset]
    io = _lib.CbLayerIO
    assert [int(x) for x in r["layer_io"]] == [ctypes.sizeof(io), io.cand.offset, io.out.offset]
