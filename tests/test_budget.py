"""Shared-memory / tensor-memory budget solver ("Warp-specialised W4A4 kernel",
section 6): per-CTA accounting of every split-or-replicate decision, checked by
a host C++ program that includes the kernel's own budget header."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp8_quantized_gemm_q4_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "budget.hpp"
using namespace bsk;
int main() {
  constexpr int misc = 2048 + 1025 * 4 + 1024;
  constexpr Fp4TileShape one{128, 256, 256, 1, true, 32, misc};
  constexpr Fp4TileShape one_nl{128, 256, 256, 1, false, 32, misc};
  constexpr Fp4TileShape pair{128, 256, 256, 2, true, 32, misc};
  // 2-CTA pair with the page's bug: up-projection block counted in full per CTA
  constexpr int split = fp4_lora_bytes(pair), repl = fp4_lora_bytes_replicated(pair);
  constexpr int stages_split = max_main_stages(round_up(fp4_stage_bytes(pair), kAlign), round_up(split, kAlign), misc);
  constexpr int stages_repl = max_main_stages(round_up(fp4_stage_bytes(pair), kAlign), round_up(repl, kAlign), misc);
  static_assert(split < repl, "split accounting must be smaller");
  constexpr int kmisc = 2048 + 1024 + 8 * 32 * 32;
  constexpr Fp4TileShape kpair{128, 256, 256, 2, true, 32, kmisc};
  constexpr int kstages_split = fp4_main_stages(kpair);
  constexpr int kstages_repl =
      max_main_stages(round_up(fp4_stage_bytes(kpair), kAlign), round_up(fp4_lora_bytes_replicated(kpair), kAlign), kmisc);
  printf("stage_one %d\n", fp4_stage_bytes(one));
  printf("stage_pair %d\n", fp4_stage_bytes(pair));
  printf("lora_one %d\n", fp4_lora_bytes(one));
  printf("lora_pair_split %d\n", split);
  printf("lora_pair_repl %d\n", repl);
  printf("stages_one %d\n", fp4_main_stages(one));
  printf("stages_one_nolora %d\n", fp4_main_stages(one_nl));
  printf("stages_pair_split %d\n", stages_split);
  printf("stages_pair_repl %d\n", stages_repl);
  printf("kernel_stages_split %d\n", kstages_split);
  printf("kernel_stages_repl %d\n", kstages_repl);
  printf("smem_one %d\n", fp4_smem_total(one, fp4_main_stages(one)));
  printf("smem_one_nolora %d\n", fp4_smem_total(one_nl, fp4_main_stages(one_nl)));
  printf("tmem_one %d\n", fp4_tmem_cols(one, 1, 2));
  printf("tmem_pow2 %d\n", pow2_cols(fp4_tmem_cols(one, 1, 2)));
  printf("tmem_double_acc %d\n", fp4_tmem_cols(one, 2, 2));
  return 0;
}
"""


@pytest.fixture(scope="module")
def budget(tmp_path_factory):
    d = tmp_path_factory.mktemp("budget")
    src = d / "budget_test.cpp"
    src.write_text(PROGRAM)
    exe = d / "budget_test"
    subprocess.check_call(["g++", "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True)
    return {k: int(v) for k, v in (line.split() for line in out.splitlines())}


def test_stage_bytes_per_cta(budget):
    # A 128x256 fp4 = 16 KiB, B 256x256 fp4 = 32 KiB, scales 2 + 4 KiB
    assert budget["stage_one"] == 16384 + 32768 + 2048 + 4096
    # a CTA of a pair holds half of B (split) but all B scale rows (replicated)
    assert budget["stage_pair"] == 16384 + 16384 + 2048 + 4096


def test_lora_split_vs_replicated(budget):
    assert budget["lora_one"] == 128 * 64 * 2 + 256 * 32 * 2
    assert budget["lora_pair_split"] == 128 * 64 * 2 + 128 * 32 * 2
    assert budget["lora_pair_repl"] - budget["lora_pair_split"] == 128 * 32 * 2


def test_stage_solver_fits_and_is_maximal(budget):
    assert budget["stages_one"] == 3 and budget["stages_one_nolora"] == 4
    assert budget["smem_one"] + 1024 <= 232448
    assert budget["smem_one_nolora"] + 1024 <= 232448
    # one more stage would not fit
    assert budget["smem_one"] + budget["stage_one"] > 232448 - 1024
    # the page's split-or-replicate decision (section 6): counting each CTA's
    # half of the up-projection block gives the pair five main stages;
    # counting the whole block in every CTA (the page's bug) gives four
    assert budget["stages_pair_split"] == 5
    assert budget["stages_pair_repl"] == 4
    # the same decision with the pair kernel's own low-rank shape (its misc
    # bytes: barriers 3 KiB + eight 32 x 32-byte output staging boxes)
    assert budget["kernel_stages_split"] == 5
    assert budget["kernel_stages_repl"] == 4


def test_tmem_budget(budget):
    assert budget["tmem_one"] == 256 + 2 * 4 * 12
    assert budget["tmem_pow2"] == 512
    assert budget["tmem_double_acc"] > 512   # why the accumulator is single-buffered at N = 256
