"""Shared test helpers: build/load the library once per session."""
import re
import os

import ring_attention_slope_gb300 as slope

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "slope.h")


def built_lib():
    slope.build()
    return slope.load()


def declared_symbols():
    """Function names declared with SLOPE_API in include/slope.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SLOPE_API\s+[\w\s\*]+?\b(slope_\w+)\s*\(", text)))
