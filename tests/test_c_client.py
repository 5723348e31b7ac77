"""The public header as a C11 client sees it: `tests/c_client/client.c` is compiled with
gcc -std=c11 -Wall -Werror against include/csa2.h, linked against libcsa2.so, and run; it
checks host-side answers that need no GPU (argument checks before any launch, size
queries, status strings)."""
import os
import subprocess
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c11_client_compiles_links_and_runs():
    from fp4_compressed_sparse_03_b300 import build
    lib = build.build()
    libdir = os.path.dirname(lib)
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "client")
        subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                               "-I", os.path.join(ROOT, "include"),
                               os.path.join(ROOT, "tests", "c_client", "client.c"),
                               "-L", libdir, "-l:libcsa2.so", "-Wl,-rpath," + libdir,
                               "-o", exe])
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        assert r.returncode == 0, r.stderr
        assert r.stdout.strip() == "ok"
