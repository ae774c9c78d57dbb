// rope_table.cuh -- builds the RoPE cos/sin table on the device.
//
// table[pos][0][i] = cos(pos * base^(-2i/hd)), table[pos][1][i] = sin(...),
// for pos in [0, npos), i < hd/2.  The angle and both functions are evaluated
// in fp64 (the double-precision CUDA math functions) and rounded once to
// fp32, so a large position does not lose the angle to fp32 rounding of
// pos * inv_freq.  Runs once per table size; not on the hot path.
#pragma once

extern "C" __global__ void rope_table_build(float* table, long long npos, int hd, double base) {
  const int half = hd / 2;
  const long long total = npos * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long pos = idx / half;
    const int i = static_cast<int>(idx % half);
    const double theta = static_cast<double>(pos) * pow(base, -2.0 * i / hd);
    double s, c;
    sincos(theta, &s, &c);
    table[pos * 2 * half + i] = static_cast<float>(c);
    table[pos * 2 * half + half + i] = static_cast<float>(s);
  }
}
