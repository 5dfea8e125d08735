"""AddressSanitizer and UndefinedBehaviorSanitizer on the host code (CPU only, no GPU work):

* the CPU oracle, on small random problems with corrupted ids and offsets (repair, forward,
  backward, the gradient with respect to per-sample weights, routing, every 16-bit pattern through
  the conversions), with leak checking;
* the CUDA library's host code (problem planner, argument validation, workspace layout, the
  no-alloc entry point), compiled with the sanitizers and linked with the library's kernel
  objects, on the paths that return before any device work.

Each program aborts on the first invalid access or undefined behaviour and prints "sanitize ok"."""
import os
import shutil
import subprocess

import pytest

from bwd_tbe_fwd_gb300 import build as tbe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.join(ROOT, "tests", "sanitize")
SAN = ["-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer"]


def _gxx_has_sanitizers(tmp_path):
    src = tmp_path / "probe.cpp"
    src.write_text("int main() { return 0; }\n")
    r = subprocess.run(["g++", *SAN, str(src), "-o", str(tmp_path / "probe")], capture_output=True)
    return r.returncode == 0


def _run(exe, env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and "sanitize ok" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])


def test_oracle_under_asan_and_ubsan(tmp_path):
    if shutil.which("g++") is None or not _gxx_has_sanitizers(tmp_path):
        pytest.skip("g++ with AddressSanitizer/UndefinedBehaviorSanitizer runtimes is not available")
    exe = tmp_path / "san_oracle"
    subprocess.run(["g++", "-std=c++17", "-O1", "-g", "-ffp-contract=off", *SAN, "-I", os.path.join(ROOT, "oracle"),
                    os.path.join(ROOT, "oracle", "tbe_oracle.cpp"), os.path.join(HERE, "sanitize_oracle.cpp"),
                    "-o", str(exe)], check=True)
    _run(exe, {"ASAN_OPTIONS": "detect_leaks=1", "UBSAN_OPTIONS": "print_stacktrace=1"})


def test_library_host_code_under_asan_and_ubsan(tmp_path):
    if shutil.which("g++") is None or not _gxx_has_sanitizers(tmp_path):
        pytest.skip("g++ with AddressSanitizer/UndefinedBehaviorSanitizer runtimes is not available")
    tbe_build.build()  # the kernel objects in the build directory
    nvcc = tbe_build._nvcc()
    xsan = ["-Xcompiler", ",".join(["-fPIC", *SAN])]
    inc = ["-I", tbe_build.INCLUDE, "-I", tbe_build.CSRC]
    host_units = ("tbe_api.cu", "tbe_noalloc.cu")
    objs = []
    for unit in host_units:
        obj = tmp_path / (unit[:-3] + ".o")
        subprocess.run([nvcc, *tbe_build.ARCH, "-O1", "-g", "-std=c++17", "--expt-relaxed-constexpr", *xsan, *inc,
                        "-c", os.path.join(tbe_build.CSRC, unit), "-o", str(obj)], check=True)
        objs.append(str(obj))
    main_obj = tmp_path / "main.o"
    subprocess.run(["g++", "-std=c++17", "-O1", "-g", *SAN, "-I", tbe_build.INCLUDE, "-c",
                    os.path.join(HERE, "sanitize_library.cpp"), "-o", str(main_obj)], check=True)
    kernels = [os.path.join(tbe_build.BUILD_DIR, f) for f in sorted(os.listdir(tbe_build.BUILD_DIR))
               if f.endswith(".o") and f[:-2] + ".cu" not in host_units]
    exe = tmp_path / "san_library"
    subprocess.run([nvcc, *tbe_build.ARCH, "-Xcompiler", ",".join(SAN[:2]), "-o", str(exe), str(main_obj), *objs,
                    *kernels, "-cudart", "shared"], check=True)
    # protect_shadow_gap=0: the CUDA driver, where one is installed, maps memory in the gap
    _run(exe, {"ASAN_OPTIONS": "protect_shadow_gap=0:detect_leaks=0", "UBSAN_OPTIONS": "print_stacktrace=1"})
