"""The square root of the PN-Mix pair norms (csrc/sqrt_rn.h) against the
CUDA runtime's correctly rounded __fsqrt_rn, bit for bit, on every
non-negative fp32 bit pattern: the straight-line path wherever it reports
itself sure, the runtime elsewhere.  A small CUDA program is compiled for
sm_103a and run on the GPU; it counts mismatches and the inputs the fast
path left to the runtime (zero, infinity and NaN only)."""
import pathlib
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

CSRC = pathlib.Path(__file__).resolve().parents[1] / "bit_kv_cache_kvq_gb300" / "csrc"

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "sqrt_rn.h"

__global__ void check(unsigned long long* bad, unsigned* first, unsigned long long* unsure) {
  const uint32_t stride = gridDim.x * blockDim.x;
  unsigned long long n = 0, nu = 0;
  for (uint32_t b = blockIdx.x * blockDim.x + threadIdx.x; b < 0x80000000u; b += stride) {
    const float s = __uint_as_float(b);
    const float want = __fsqrt_rn(s);
    const float got = sqrt_rn(s);
    bool sure;
    sqrt_rn_fast(s, sure);
    nu += sure ? 0 : 1;
    const bool same = __float_as_uint(got) == __float_as_uint(want) || (want != want && got != got);
    if (!same) {
      ++n;
      atomicMin(first, b);
    }
  }
  if (n) atomicAdd(bad, n);
  if (nu) atomicAdd(unsure, nu);
}

int main() {
  unsigned long long *bad, *unsure;
  unsigned* first;
  cudaMalloc(&bad, sizeof(*bad));
  cudaMalloc(&unsure, sizeof(*unsure));
  cudaMalloc(&first, sizeof(*first));
  cudaMemset(bad, 0, sizeof(*bad));
  cudaMemset(unsure, 0, sizeof(*unsure));
  cudaMemset(first, 0xff, sizeof(*first));
  check<<<152 * 8, 256>>>(bad, first, unsure);
  unsigned long long h = 0, u = 0;
  unsigned f = 0;
  cudaError_t e = cudaMemcpy(&h, bad, sizeof(h), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&u, unsure, sizeof(u), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&f, first, sizeof(f), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    std::printf("cuda error %s\n", cudaGetErrorString(e));
    return 2;
  }
  std::printf("mismatches %llu first 0x%08x unsure %llu\n", h, f, u);
  return h == 0 ? 0 : 1;
}
"""


def test_sqrt_rn_matches_runtime_on_every_nonnegative_float(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    src = tmp_path / "check_sqrt.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "check_sqrt"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-I", str(CSRC),
                    str(src), "-o", str(exe)], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0 " in r.stdout
    # the runtime takes exactly +0, +inf and the 2^23 - 1 positive NaN
    # patterns; every positive finite input (subnormals too) runs straight
    unsure = int(r.stdout.split("unsure")[1])
    assert unsure == (1 << 23) + 1, r.stdout
