"""Host checks of the packed-code bit layout (csrc/frag_layout.h).

The header is compiled with g++ (no GPU) into a small checker that
verifies, for 2- and 4-bit keys and values:
  * the forward map (token, channel) -> (word, bit) is a bijection onto the
    code section's bits, with every code inside its word;
  * the inverse map (word, slot) -> (token, channel) undoes it;
  * the code of every mma.sync A-fragment element sits where the decode
    kernel's unpack reads it: register a_r of (tile, k, lane) taken from
    x (r even) or x >> 8 (r odd), masked at the bit position the layout
    assigns to (k & 1, r >> 1).
"""
import pathlib
import shutil
import subprocess

import pytest

CSRC = pathlib.Path(__file__).resolve().parents[1] / "bit_kv_cache_kvq_gb300" / "csrc"

CHECKER = r"""
#include <cstdio>
#include <vector>
#include "frag_layout.h"
using namespace kvq;

static int fail = 0;
#define CHECK(c, ...) do { if (!(c)) { if (fail < 10) std::printf(__VA_ARGS__); ++fail; } } while (0)

// bit of element (row, col) of A fragment register `reg` as the kernel reads it
static int kernel_bit(int bits, int k, int reg, int half) {
  const int from_y = reg & 1;            // a1, a3 come from x >> 8
  const int pos = bits == 2 ? 2 * (2 * (k & 1) + (reg >> 1)) : 4 * (reg >> 1);
  return pos + 8 * from_y + 16 * half;
}

static void check(int bits, bool key) {
  const int words = 128 * 128 * bits / 32;
  std::vector<int> seen(words * 32, 0);
  for (int tok = 0; tok < 128; ++tok)
    for (int ch = 0; ch < 128; ++ch) {
      const CodePos p = key ? key_code_pos(tok, ch, bits) : value_code_pos(tok, ch, bits);
      CHECK(p.word >= 0 && p.word < words, "word out of range %d\n", p.word);
      CHECK(p.bit >= 0 && p.bit + bits <= 32 && p.bit % bits == 0, "bad bit %d\n", p.bit);
      if (p.word < 0 || p.word >= words || p.bit < 0 || p.bit > 31) continue;
      for (int b = 0; b < bits; ++b) ++seen[p.word * 32 + p.bit + b];
      int t2 = -1, c2 = -1;
      if (key) key_word_code(p.word, p.bit / bits, bits, t2, c2);
      else value_word_code(p.word, p.bit / bits, bits, t2, c2);
      CHECK(t2 == tok && c2 == ch, "inverse (%d,%d) -> (%d,%d)\n", tok, ch, t2, c2);
      // fragment coordinates: keys have rows = tokens, values rows = channels
      int tile, k, lane, reg, half;
      if (key) frag_coords(tok, ch, tile, k, lane, reg, half);
      else frag_coords(ch, tok, tile, k, lane, reg, half);
      CHECK(p.bit == kernel_bit(bits, k, reg, half), "kernel bit %d vs %d\n", p.bit,
            kernel_bit(bits, k, reg, half));
      // a lane's words: the kernel reads word(tile, k-pair, lane) at lane stride 1
      // (keys 2-bit), 2 (keys 4-bit) or 4 (values)
      const int stride = key ? (bits == 2 ? 1 : 2) : 4;
      CHECK((p.word / stride) % 32 == lane, "lane %d word %d\n", lane, p.word);
    }
  for (int i = 0; i < words * 32; ++i) CHECK(seen[i] == 1, "bit %d covered %d times\n", i, seen[i]);
}

int main() {
  for (int bits : {2, 4}) {
    check(bits, true);
    check(bits, false);
  }
  std::printf("%s %d\n", fail ? "FAIL" : "OK", fail);
  return fail ? 1 : 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="g++ not available")
def test_frag_layout_bijective_and_matches_unpack(tmp_path):
    src = tmp_path / "check.cpp"
    src.write_text(CHECKER)
    exe = tmp_path / "check"
    subprocess.run(["g++", "-O1", "-std=c++17", "-D__host__=", "-D__device__=", f"-I{CSRC}",
                    str(src), "-o", str(exe)], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("OK")
