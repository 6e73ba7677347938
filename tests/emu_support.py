"""Building the CPU block emulator's harnesses (tests/emu/): the host
compiler command, with AddressSanitizer when the toolchain has it, so that
a kernel source that reads or writes past a buffer fails its test the way it
would fault on a GPU."""
import functools
import shutil
import subprocess
import tempfile
from pathlib import Path

import pytest

EMU = Path(__file__).resolve().parent / "emu"
BASE = ["-std=c++20", "-O2", "-pthread", "-Wno-unknown-pragmas"]
ASAN = ["-fsanitize=address", "-fno-omit-frame-pointer"]


@functools.lru_cache(maxsize=1)
def asan_flags() -> tuple:
    if shutil.which("g++") is None:
        return ()
    with tempfile.TemporaryDirectory() as d:
        src = Path(d) / "t.cpp"
        src.write_text("int main() { return 0; }\n")
        r = subprocess.run(["g++", *ASAN, str(src), "-o", str(Path(d) / "t")], capture_output=True)
        if r.returncode != 0:
            return ()
        r = subprocess.run([str(Path(d) / "t")], capture_output=True)
        return tuple(ASAN) if r.returncode == 0 else ()


def compile_harness(main_cpp: str, include_dir: Path, exe: Path):
    """g++ the harness main (tests/emu/<main_cpp>) with the kernel source in
    include_dir; fails the test with the compiler's message."""
    if shutil.which("g++") is None:
        pytest.skip("no host C++ compiler")
    r = subprocess.run(["g++", *BASE, *asan_flags(), "-I", str(EMU), "-I", str(include_dir),
                        str(EMU / main_cpp), "-o", str(exe)], capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    return exe


class EmulatorFault(AssertionError):
    """The emulated kernel stopped on one of the emulator's own checks (a
    barrier protocol or shared-memory rule broken, an AddressSanitizer
    report) instead of finishing."""


def check_run(r):
    """Raise EmulatorFault with the emulator's message when its run failed."""
    if r.returncode != 0:
        raise EmulatorFault(r.stderr[-2000:])


def rejected(run):
    """For a planted mistake: True when run() raises EmulatorFault from one of
    the emulator's checks, else run()'s own verdict (a result outside the
    tolerance must be reported as True by run)."""
    try:
        return run()
    except EmulatorFault as e:
        msg = str(e)
        return "emulator:" in msg or "AddressSanitizer" in msg
