"""Helpers shared by the tests: build/load the CUDA library and list the
entry points that include/sq.h declares."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sq.h")


def ensure_built():
    from w8a8_post_quantization_02_b300 import build_lib
    return build_lib.build()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sq_[a-z0-9_]+)\s*\(", text)))
