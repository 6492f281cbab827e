"""Every environment variable the library reads is documented in the
header's Environment block, and every variable documented there is read by
the library (no stale names on either side)."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "collective_all_reduce_rank_gb300", "csrc")
HEADER = os.path.join(ROOT, "include", "rra.h")


def _read_by_library():
    names = set()
    for f in os.listdir(CSRC):
        if f.endswith((".cpp", ".cu", ".cuh", ".h")):
            text = open(os.path.join(CSRC, f)).read()
            names |= set(re.findall(r'"(RRA_[A-Z0-9_]+)"', text))
    return names


def _documented():
    """RRA_ names in the Environment block, less the header's own constants
    (enumerators and macros the text mentions)."""
    text = open(HEADER).read()
    start = text.index("Environment (read by the library")
    block = text[start:text.index("*/", start)]
    constants = set(re.findall(r"\b(RRA_[A-Z0-9_]+)\s*=", text)) | set(re.findall(r"#define\s+(RRA_[A-Z0-9_]+)", text))
    return set(re.findall(r"\bRRA_[A-Z0-9_]+\b", block)) - constants


def test_every_variable_read_is_documented():
    missing = _read_by_library() - _documented()
    assert not missing, sorted(missing)


def test_every_documented_variable_is_read():
    stale = _documented() - _read_by_library()
    assert not stale, sorted(stale)
