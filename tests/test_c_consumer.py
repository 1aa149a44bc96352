"""The C ABI from plain C: a C11 program includes include/jfa.h, links against
libjfa.so and calls the entry points that need no GPU (status strings, the
host planners, argument rejection before any device work).  CPU only."""
import os
import shutil
import subprocess

import pytest

from variable_length_attention_gb300 import jfa as J

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "jfa.h"

int main(void) {
  /* the jagged layout's worked example (n1n.ai page on JFA with TLX): lengths 128, 4096, 512, 2048 */
  const int32_t offsets[5] = {0, 128, 4224, 4736, 6784};
  int32_t units[4 * 64], cta_start[5];
  const int n = jfa_plan_fwd(offsets, 4, 1, 0, 0, 4, units, cta_start);
  printf("fwd_units %d\n", n);
  printf("cta_start %d %d %d %d %d\n", cta_start[0], cta_start[1], cta_start[2], cta_start[3], cta_start[4]);
  printf("first_unit %d %d %d %d\n", units[0], units[1], units[2], units[3]);
  printf("bwd_units %d\n", jfa_plan_bwd(offsets, 4, 1, 0, 0, 4, NULL, NULL));
  int32_t bpb[5], prog[9];
  printf("block_programs %d\n", block_plan(offsets, 4, 1, 8, bpb, prog));
  printf("block_prefix %d %d %d %d %d\n", bpb[0], bpb[1], bpb[2], bpb[3], bpb[4]);
  printf("status %s\n", jfa_status_string(JFA_ERR_BAD_OFFSETS));
  /* rejected before any device work: head_dim 96 */
  static char fake[256];
  static int32_t fake_offsets[5];
  printf("reject %d\n", jfa_fwd(fake, fake, fake, fake, NULL, fake_offsets, offsets, 4, 4096, 0, 2, 2, 96, 0.1f, 0,
                                0, fake, sizeof fake, NULL));
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_uses_the_abi(tmp_path):
    lib = J.load()._name  # built in-tree
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                           lib, "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60, check=True).stdout
    got = dict(line.split(" ", 1) for line in out.strip().splitlines())
    # 256-row forward units: 1 + 16 + 2 + 8 = 27; 128-key backward units: 1 + 32 + 4 + 16 = 53
    assert got["fwd_units"] == "27" and got["bwd_units"] == "53"
    assert got["cta_start"] == "0 7 14 21 27"   # 27 units snake-dealt over 4 CTAs: 7, 7, 7, 6
    assert got["first_unit"] == "1 0 0 32"      # the largest cost first: sequence 1, 4096 keys = 32 blocks
    assert got["block_programs"] == "8"
    assert got["block_prefix"] == "0 2 66 74 106"  # 64-token blocks per sequence: 2, 64, 8, 32
    assert got["status"] == "bad offsets"
    assert got["reject"] == "2"                 # JFA_ERR_UNSUPPORTED
