"""include/slope.h is valid C99 on its own, and the binding's ctypes structures and
constants match it field by field (sizes and offsets as a C compiler lays them out)."""
import ctypes
import os
import subprocess

import pytest

import ring_attention_slope_gb300 as slope

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")

PROBE = r"""
#include <stddef.h>
#include <stdio.h>
#include "slope.h"
#define F(T, f) printf(#T "." #f " %zu %zu\n", offsetof(T, f), sizeof(((T*)0)->f));
int main(void) {
  printf("slope_tensor %zu\n", sizeof(slope_tensor));
  F(slope_tensor, data) F(slope_tensor, dtype) F(slope_tensor, ndim) F(slope_tensor, shape) F(slope_tensor, stride)
  printf("slope_plan_item %zu\n", sizeof(slope_plan_item));
  F(slope_plan_item, launch) F(slope_plan_item, plane) F(slope_plan_item, q_row0) F(slope_plan_item, q_len)
  F(slope_plan_item, n_kv) F(slope_plan_item, kv_row0) F(slope_plan_item, kv_len) F(slope_plan_item, head_group)
  F(slope_plan_item, n_head_groups)
  printf("layouts %d %d %d %d\n", SLOPE_LAYOUT_CONTIGUOUS, SLOPE_LAYOUT_ZIGZAG, SLOPE_LAYOUT_CHUNKED,
         SLOPE_LAYOUT_ULYSSES);
  printf("dtypes %d %d\n", SLOPE_BF16, SLOPE_F32);
  printf("flags %u\n", SLOPE_CP_BF16_PARTIALS);
  {
    slope_layout l = (slope_layout)(SLOPE_LAYOUT_ZIGZAG | SLOPE_ULYSSES_DEGREE(4));
    printf("layout_word %d\n", (int)l);
  }
  return 0;
}
"""


def test_header_compiles_as_c99_and_matches_the_binding(tmp_path):
    src = tmp_path / "probe.c"
    exe = tmp_path / "probe"
    src.write_text(PROBE)
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", HEADER_DIR,
                           str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True).splitlines()
    got = {}
    for line in out:
        key, *vals = line.split()
        got[key] = [int(x) for x in vals]
    for cname, cls in (("slope_tensor", slope.SlopeTensor), ("slope_plan_item", slope.SlopePlanItem)):
        assert got[cname] == [ctypes.sizeof(cls)], cname
        for fname, _ in cls._fields_:
            field = getattr(cls, fname)
            assert got[f"{cname}.{fname}"] == [field.offset, field.size], f"{cname}.{fname}"
    assert got["layouts"] == [slope.LAYOUTS[k] for k in ("contiguous", "zigzag", "chunked", "ulysses")]
    assert got["dtypes"] == [0, 1]
    assert got["flags"] == [slope.CP_BF16_PARTIALS]
    assert got["layout_word"] == [slope.layout_code("zigzag", 4)]
