"""The C ABI used from C, without Python: include/tfm.h compiles as strict C99
and as C++17, and a C program linked against libtfm.so validates configs and
sizes its buffers on the host (no GPU needed), with the same answers the Python
binding gets from the same library."""
import os
import shutil
import subprocess

import pytest

import workloads
from decoder_only_transformer_gb300 import _build, tfm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include "tfm.h"

int main(void) {
    tfm_config cfg = {.vocab = %(vocab)d, .d_model = %(d_model)d, .n_head = %(n_head)d,
                      .n_kv_head = %(n_kv_head)d, .n_layer = %(n_layer)d, .d_ff = %(d_ff)d,
                      .max_seq = %(seq)d, .max_batch = %(batch)d, .rope_theta = 10000.0f,
                      .norm_eps = 1e-5f, .mode = TFM_BF16};
    void* handle = NULL;
    printf("abi %%d\n", (int)tfm_abi_version());
    printf("valid %%d\n", (int)tfm_validate_config(&cfg));
    printf("workspace %%zu\n", tfm_workspace_bytes(&cfg));
    printf("weights %%zu\n", tfm_weight_bytes(&cfg));
    printf("create_null_handle %%d\n", (int)tfm_create(&cfg, NULL));
    cfg.n_kv_head = 3;
    printf("group3 %%d %%s\n", (int)tfm_validate_config(&cfg), tfm_last_error());
    tfm_destroy(handle);
    return 0;
}
"""


def _compiler(name):
    path = shutil.which(name)
    if path is None:
        pytest.skip(f"{name} not installed")
    return path


@pytest.mark.parametrize("std", ["-std=c99", "-std=c11"])
def test_header_is_strict_c(tmp_path, std):
    src = tmp_path / "only_header.c"
    src.write_text('#include "tfm.h"\nint main(void) { return tfm_abi_version() == 1 ? 0 : 1; }\n')
    r = subprocess.run([_compiler("gcc"), std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE,
                        "-c", str(src), "-o", str(tmp_path / "o.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_header_is_cxx(tmp_path):
    src = tmp_path / "only_header.cc"
    src.write_text('#include "tfm.h"\nint main() { return tfm_abi_version() == 1 ? 0 : 1; }\n')
    r = subprocess.run([_compiler("g++"), "-std=c++17", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", INCLUDE, "-c", str(src), "-o", str(tmp_path / "o.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_and_agrees_with_the_binding(tmp_path):
    cfg = workloads.get_config("gqa")
    lib = tfm.load()
    libdir = os.path.dirname(_build.LIB)
    src = tmp_path / "main.c"
    src.write_text(PROGRAM % dict(vocab=cfg.vocab, d_model=cfg.d_model, n_head=cfg.n_head,
                                  n_kv_head=cfg.n_kv_head, n_layer=cfg.n_layer, d_ff=cfg.d_ff,
                                  seq=cfg.seq, batch=cfg.batch))
    exe = tmp_path / "main"
    r = subprocess.run([_compiler("gcc"), "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, str(src),
                        "-L", libdir, "-ltfm", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    got = dict(line.split(" ", 1) for line in out.stdout.strip().splitlines())
    c = tfm.make_config(cfg)
    assert int(got["abi"]) == lib.tfm_abi_version()
    assert int(got["valid"]) == tfm.TFM_OK
    assert int(got["workspace"]) == tfm.workspace_bytes(c)
    assert int(got["weights"]) == tfm.weight_bytes(c)
    assert int(got["create_null_handle"]) == tfm.TFM_EINVAL
    status, msg = got["group3"].split(" ", 1)
    assert int(status) == tfm.TFM_EINVAL and "n_kv_head" in msg
