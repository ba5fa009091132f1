"""The boundary as a C caller sees it (no GPU needed).

include/q4nx.h compiles as strict C99 and as C++17 without warnings, and a C
program built against it links with libq4nx.so and gets the documented
answers from calls that are settled on the host: chunk sizes of the chunk-kind
table (the "Q4NX chunks" section of the 1bit engine "NPU engine" page), the
ABI version, and the refusals of a NULL weight, an unknown chunk kind and a
row count that is not a multiple of 32, each before any device work.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include "q4nx.h"
#include <stdio.h>

int main(void) {
    q4nx_weight w;
    unsigned long long sizes[5];
    int k;
    for (k = 0; k < 5; ++k) sizes[k] = (unsigned long long)q4nx_chunk_bytes(k);
    printf("chunk_bytes %llu %llu %llu %llu %llu\n", sizes[0], sizes[1], sizes[2], sizes[3], sizes[4]);
    printf("abi %d\n", q4nx_abi_version());
    printf("null_weight %d\n", q4nx_gemv(NULL, NULL, NULL, Q4NX_OUT_BF16, NULL, 0, NULL));
    w.chunks_dev = (const void*)0x100000;   /* never dereferenced: refused on the host */
    w.bytes = 5120;
    w.kind = 7;
    w.reserved = 0;
    w.rows = 32;
    w.cols = 256;
    printf("unknown_kind %d\n", q4nx_decode(&w, (void*)0x200000, 1u << 20, NULL));
    w.kind = Q4NX_Q4_1;
    w.rows = 33;
    printf("bad_rows %d %llu\n", q4nx_decode(&w, (void*)0x200000, 1u << 20, NULL),
           (unsigned long long)q4nx_gemv_workspace(&w));
    printf("status_str %s\n", q4nx_status_str(Q4NX_E_SHAPE));
    return 0;
}
"""


@pytest.fixture(scope="module")
def lib_dir():
    import __graft_entry__

    __graft_entry__._load_build_module().build()
    import dequant_gemv_gb300

    return os.path.dirname(dequant_gemv_gb300.LIB_PATH)


def _compiler(name):
    path = shutil.which(name)
    if path is None:
        pytest.skip(f"{name} not installed")
    return path


def test_header_compiles_as_c99_and_cpp17():
    inc = os.path.join(ROOT, "include")
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "h.c")
        with open(c, "w") as f:
            f.write('#include "q4nx.h"\nint q4nx_header_probe(void) { return Q4NX_OK; }\n')
        subprocess.run([_compiler("gcc"), "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", inc,
                        "-c", c, "-o", os.path.join(d, "h.o")], check=True)
        cc = os.path.join(d, "h.cpp")
        with open(cc, "w") as f:
            f.write('#include "q4nx.h"\nint q4nx_header_probe_cpp() { return Q4NX_OK; }\n')
        subprocess.run([_compiler("g++"), "-std=c++17", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", inc,
                        "-c", cc, "-o", os.path.join(d, "hpp.o")], check=True)


def test_c_program_links_and_gets_host_side_answers(lib_dir):
    inc = os.path.join(ROOT, "include")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "prog.c"), os.path.join(d, "prog")
        with open(src, "w") as f:
            f.write(PROGRAM)
        subprocess.run([_compiler("gcc"), "-std=c99", "-Wall", "-Werror", "-I", inc, src, "-o", exe,
                        "-L", lib_dir, "-lq4nx", "-Wl,-rpath," + lib_dir], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split("\n")
    got = dict(line.split(" ", 1) for line in out if line)
    assert got["chunk_bytes"] == "0 5120 4736 8704 8704"
    assert got["abi"] == "1"
    assert got["null_weight"] == "1"          # Q4NX_E_NULL
    assert got["unknown_kind"] == "2"         # Q4NX_E_KIND
    assert got["bad_rows"] == "3 0"           # Q4NX_E_SHAPE, and no workspace size for it
    assert got["status_str"] != "unknown status"
