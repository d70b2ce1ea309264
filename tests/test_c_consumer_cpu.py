"""The C ABI from plain C (no GPU needed): a C99 program that includes include/kda.h compiles with
-std=c99 -pedantic -Wall -Wextra -Werror, links against libkda.so, and its host-side calls return
the documented results: the defaults, the status strings, the workspace size, and the argument
checks that return before any work is enqueued (no pointer passed is ever dereferenced).  The
program also reports the layout of kda_params, which the Python binding's ctypes mirror must
match field by field."""
import ctypes
import os
import shutil
import subprocess

import pytest

from kda_gated_delta_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stddef.h>
#include <stdio.h>
#include <string.h>
#include "kda.h"

#define EXPECT(cond, code) do { if (!(cond)) { printf("failed: %s\n", #cond); return code; } } while (0)

int main(void)
{
    kda_params p;
    size_t ws;
    int32_t rc;
    /* 16-byte aligned dummy addresses: the checks below return before any of them is used */
    void* const dev = (void*)(size_t)(1u << 20);
    float* const f = (float*)dev;
    int32_t* const idx = (int32_t*)dev;

    kda_params_init(&p, 32, 128);
    EXPECT(p.num_heads == 32 && p.head_dim == 128 && p.chunk_size == 64, 1);
    EXPECT(p.io_dtype == KDA_BF16 && p.out_dtype == KDA_BF16 && p.gate_kind == KDA_GATE_PER_CHANNEL, 2);
    EXPECT(p.use_lower_bound == 0 && p.scale == 0.0f && p.softplus_threshold == 20.0f, 3);
    EXPECT(strlen(kda_status_string(KDA_OK)) > 0 && strlen(kda_status_string(12345)) > 0, 4);

    /* one 74,240-byte record per (chunk, head) for 2 x 32 chunks of 64 tokens, plus the table */
    ws = kda_chunk_prefill_workspace_size(&p, 2, 4096);
    EXPECT(ws >= (size_t)64 * 32 * 74240, 5);

    /* rejected on the host, nothing enqueued */
    rc = kda_recurrent_decode(&p, NULL, dev, dev, f, f, f, NULL, 4, f, 8, idx, dev, NULL);
    EXPECT(rc == KDA_ERR_INVALID_ARG, 6);
    rc = kda_recurrent_decode(&p, (char*)dev + 4, dev, dev, f, f, f, NULL, 4, f, 8, idx, dev, NULL);
    EXPECT(rc == KDA_ERR_MISALIGNED, 7);
    p.head_dim = 48;
    rc = kda_recurrent_decode(&p, dev, dev, dev, f, f, f, NULL, 4, f, 8, idx, dev, NULL);
    EXPECT(rc == KDA_ERR_UNSUPPORTED, 8);
    p.head_dim = 128;
    rc = kda_chunk_prefill(&p, dev, dev, dev, f, f, f, NULL, idx, 2, 4096, f, 8, idx, dev,
                           dev, 1024, NULL);
    EXPECT(rc == KDA_ERR_WORKSPACE, 9);
    rc = kda_recurrent_verify(&p, dev, dev, dev, f, f, f, NULL, 4, 17, f, 8, idx, f, dev, NULL);
    EXPECT(rc == KDA_ERR_INVALID_ARG, 10);

    /* the struct layout, for the comparison with the Python binding's mirror */
    printf("layout %zu", sizeof(kda_params));
    printf(" num_heads=%zu head_dim=%zu io_dtype=%zu out_dtype=%zu gate_kind=%zu chunk_size=%zu",
           offsetof(kda_params, num_heads), offsetof(kda_params, head_dim), offsetof(kda_params, io_dtype),
           offsetof(kda_params, out_dtype), offsetof(kda_params, gate_kind), offsetof(kda_params, chunk_size));
    printf(" use_lower_bound=%zu lower_bound=%zu scale=%zu l2_eps=%zu softplus_threshold=%zu\n",
           offsetof(kda_params, use_lower_bound), offsetof(kda_params, lower_bound), offsetof(kda_params, scale),
           offsetof(kda_params, l2_eps), offsetof(kda_params, softplus_threshold));
    printf("ok %zu\n", ws);
    return 0;
}
"""


@pytest.fixture(scope="module")
def lib_dir():
    return os.path.dirname(build.build())


def test_c99_program_compiles_links_and_runs(tmp_path, lib_dir):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    cmd = [gcc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", lib_dir, "-lkda", f"-Wl,-rpath,{lib_dir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = r.stdout.strip().splitlines()
    assert lines[-1].startswith("ok ")
    # the binding's ctypes mirror of kda_params has the C compiler's size and field offsets
    layout = lines[-2].split()
    assert layout[0] == "layout" and int(layout[1]) == ctypes.sizeof(binding.Params)
    for item in layout[2:]:
        name, off = item.split("=")
        assert getattr(binding.Params, name).offset == int(off), name
    assert len(layout) - 2 == len(binding.Params._fields_)
