"""The in-tree library build (ternary_weight_moe_02_b300/build_lib.py), with a stand-in
compiler: objects are cached by a hash of their source and the headers, and the library
is relinked whenever the set of objects it was linked from changes, including when a
source goes back to a version whose (older) object is still cached."""
import os
import stat
import sys

import pytest

from ternary_weight_moe_02_b300 import build_lib

# "-c src -o out" copies the source into the object; a link writes the objects' contents
# in order into the output
FAKE_NVCC = """#!{python}
import sys
args = sys.argv[1:]
out = args[args.index("-o") + 1]
if "-c" in args:
    src = args[args.index("-c") + 1]
    data = open(src).read()
else:
    objs = [a for a in args if a.endswith(".o")]
    data = "".join(open(o).read() for o in objs)
open(out, "w").write(data)
"""


@pytest.fixture
def tree(tmp_path, monkeypatch):
    csrc, inc, build = tmp_path / "csrc", tmp_path / "include", tmp_path / "_build"
    csrc.mkdir()
    inc.mkdir()
    (inc / "maple.h").write_text("header\n")
    (csrc / "a.cu").write_text("A1\n")
    (csrc / "b.cu").write_text("B1\n")
    nvcc = tmp_path / "nvcc"
    nvcc.write_text(FAKE_NVCC.format(python=sys.executable))
    nvcc.chmod(nvcc.stat().st_mode | stat.S_IEXEC)
    lib = tmp_path / "libmaple.so"
    monkeypatch.setattr(build_lib, "CSRC", str(csrc))
    monkeypatch.setattr(build_lib, "INCLUDE", str(inc))
    monkeypatch.setattr(build_lib, "BUILD", str(build))
    monkeypatch.setattr(build_lib, "LIB", str(lib))
    monkeypatch.setattr(build_lib, "NVCC", str(nvcc))
    return csrc, lib


def test_build_links_every_source_and_skips_an_unchanged_tree(tree):
    csrc, lib = tree
    build_lib.build()
    assert lib.read_text() == "A1\nB1\n"
    before = os.stat(lib).st_mtime_ns
    build_lib.build()
    assert os.stat(lib).st_mtime_ns == before  # nothing changed: no relink


def test_build_relinks_when_a_source_returns_to_a_cached_version(tree):
    csrc, lib = tree
    build_lib.build()
    (csrc / "a.cu").write_text("A2\n")
    build_lib.build()
    assert lib.read_text() == "A2\nB1\n"
    (csrc / "a.cu").write_text("A1\n")  # its object from the first build is still cached
    build_lib.build()
    assert lib.read_text() == "A1\nB1\n"


def test_build_recompiles_everything_when_a_header_changes(tree, tmp_path):
    csrc, lib = tree
    build_lib.build()
    n_objs = len(os.listdir(tmp_path / "_build"))
    (tmp_path / "include" / "maple.h").write_text("header v2\n")
    build_lib.build()
    assert len(os.listdir(tmp_path / "_build")) == 2 * n_objs
    assert lib.read_text() == "A1\nB1\n"
