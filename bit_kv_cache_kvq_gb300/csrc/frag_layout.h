// Bit layout of the packed codes inside a group record.
//
// The decode kernel multiplies codes on tensor cores with
// mma.sync.m16n8k16 (f16 operands, fp32 accumulators).  Its A operand comes
// from registers, so the codes are stored in the order the A fragments need
// them: one load per lane yields the codes of whole fragments, and one AND
// turns a pair of codes into an f16x2 register.  With every other bit of a
// 16-bit half cleared, the half is an f16 subnormal whose value is exactly
// c * 2^(pos - 24), pos being the bit of the code's least significant bit;
// the tensor cores take subnormal operands exactly, and the B rows carry the
// factor 2^(24 - pos) (times one common power of two) that cancels it.
//
// Fragment convention (lane = 4g + t):
//   A (16x16, row): a0 = A[g][2t,2t+1]  a1 = A[g+8][2t,2t+1]
//                   a2 = A[g][2t+8,+9]  a3 = A[g+8][2t+8,+9]
//   B (16x8, col):  b0 = B[2t,2t+1][g]  b1 = B[2t+8,2t+9][g]
//   C (16x8):       c0 = C[g][2t] c1 = C[g][2t+1] c2 = C[g+8][2t] c3 = C[g+8][2t+1]
//
// Key codes form A of S = C_K Q' (rows = 16 tokens of M-tile mt, columns =
// 16 channels of k-step ks); value codes form A of O^T = C_V^T P' (rows =
// 16 channels of M-tile mc, columns = 16 tokens of k-step kt).  Both use the
// same in-word layout; they differ in which index is "row".
//
// 2-bit: a 32-bit word x holds two k-steps (k_local = k & 1) of one (tile,
// lane): 8 pairs P, pair P's first code at bits 2P, second at 16 + 2P, with
//   P(k_local, reg) = 4 * (reg & 1) + 2 * k_local + (reg >> 1).
// Registers a0, a2 come from x, a1, a3 from y = x >> 8, each masked to the
// bits 2 * (2 * k_local + (reg >> 1)): a0 and a1 (which meet B rows 2t,
// 2t+1) share one bit position, a2 and a3 (B rows 2t+8, 2t+9) another.
// 4-bit: a word holds one k-step: nibble n(reg) = 2 * (reg & 1) + (reg >> 1)
// at bits 4n and 16 + 4n; a0, a2 from x masked at bits 0 and 4, a1, a3 from
// y = x >> 8 at the same bits.
//
// Word order in the 4096 B (2-bit) / 8192 B (4-bit) code section:
//   key  2-bit: word(mt, lane, w = ks/2)       = (mt*4 + w)*32 + lane
//   key  4-bit: word(mt, lane, ks)             = ((mt*4 + ks/2)*32 + lane)*2 + ks%2
//   value 2-bit: word(mc, lane, w = kt/2)      = (mc*32 + lane)*4 + w
//   value 4-bit: word(mc, lane, kt)            = ((mc*2 + kt/4)*32 + lane)*4 + kt%4
// Keys: a warp reads one word (2-bit) or two (4-bit) per lane per load, the
// k-step order of the QK loop; values: 16 bytes per lane per load, one
// channel tile over all (2-bit) or half (4-bit) of the group's token
// k-steps, the order of the P·V loop.  Every load is contiguous across the
// warp, so it is free of shared-memory bank conflicts.
#pragma once

#include <cstdint>

namespace kvq {

// Position of one code: 32-bit word index in the section and bit offset.
struct CodePos {
  int word;
  int bit;
};

// (row, col) -> fragment coordinates shared by both layouts.
__host__ __device__ inline void frag_coords(int row, int col, int& tile, int& k,
                                            int& lane, int& reg, int& half) {
  tile = row >> 4;
  k = col >> 4;
  const int r = row & 15, c = col & 15;
  const int g = r & 7, rhi = r >> 3;
  const int chi = c >> 3, t = (c & 7) >> 1;
  half = c & 1;
  lane = 4 * g + t;
  reg = rhi + 2 * chi;
}

__host__ __device__ inline int pair_2bit(int k_local, int reg) {
  return 4 * (reg & 1) + 2 * k_local + (reg >> 1);
}
__host__ __device__ inline int nibble_4bit(int reg) { return 2 * (reg & 1) + (reg >> 1); }
// Inverses: code slot (bit order within a 16-bit half) -> register.
__host__ __device__ inline int reg_of_pair(int P) { return (P >> 2) | ((P & 1) << 1); }
__host__ __device__ inline int k_local_of_pair(int P) { return (P >> 1) & 1; }
__host__ __device__ inline int reg_of_nibble(int n) { return (n >> 1) | ((n & 1) << 1); }

// Key code of token tok, channel ch (rows = tokens, columns = channels).
__host__ __device__ inline CodePos key_code_pos(int tok, int ch, int bits) {
  int mt, ks, lane, reg, half;
  frag_coords(tok, ch, mt, ks, lane, reg, half);
  if (bits == 2)
    return {(mt * 4 + (ks >> 1)) * 32 + lane, 2 * pair_2bit(ks & 1, reg) + 16 * half};
  return {((mt * 4 + (ks >> 1)) * 32 + lane) * 2 + (ks & 1), 4 * nibble_4bit(reg) + 16 * half};
}

// Mixed keys: 2-bit virtual channel v of token tok, kw2 words per (tile,
// lane) instead of 4 (the uniform 2-bit key layout is the case kw2 = 4).
__host__ __device__ inline CodePos mixed_code_pos(int tok, int v, int kw2) {
  int mt, ks, lane, reg, half;
  frag_coords(tok, v, mt, ks, lane, reg, half);
  return {(mt * kw2 + (ks >> 1)) * 32 + lane, 2 * pair_2bit(ks & 1, reg) + 16 * half};
}

// Value code of token tok, channel ch (rows = channels, columns = tokens).
__host__ __device__ inline CodePos value_code_pos(int tok, int ch, int bits) {
  int mc, kt, lane, reg, half;
  frag_coords(ch, tok, mc, kt, lane, reg, half);
  if (bits == 2)
    return {(mc * 32 + lane) * 4 + (kt >> 1), 2 * pair_2bit(kt & 1, reg) + 16 * half};
  return {((mc * 2 + (kt >> 2)) * 32 + lane) * 4 + (kt & 3), 4 * nibble_4bit(reg) + 16 * half};
}

// Inverse maps: for word w and bit position p of a code, the (row, col) it
// holds.  Used by the packer, which assembles whole words.
__host__ __device__ inline void frag_rowcol(int tile, int k, int lane, int reg, int half,
                                            int& row, int& col) {
  const int g = lane >> 2, t = lane & 3;
  row = tile * 16 + g + 8 * (reg & 1);
  col = k * 16 + 2 * t + 8 * (reg >> 1) + half;
}

// Key word w, code slot s (0..32/bits-1 in bit order) -> (tok, ch).
__host__ __device__ inline void key_word_code(int w, int s, int bits, int& tok, int& ch) {
  int tile, k, lane, reg, half;
  if (bits == 2) {
    lane = w & 31;
    const int wi = (w >> 5) & 3;
    tile = w >> 7;
    half = s >> 3;
    const int P = s & 7;  // bit 2P (+16)
    reg = reg_of_pair(P);
    k = 2 * wi + k_local_of_pair(P);
  } else {
    lane = (w >> 1) & 31;
    k = 2 * ((w >> 6) & 3) + (w & 1);
    tile = w >> 8;
    half = s >> 2;
    reg = reg_of_nibble(s & 3);
  }
  frag_rowcol(tile, k, lane, reg, half, tok, ch);
}

// Mixed key word w, code slot s -> (tok, virtual channel v).
__host__ __device__ inline void mixed_word_code(int w, int s, int kw2, int& tok, int& v) {
  const int lane = w & 31, q = w >> 5;
  const int tile = q / kw2, wi = q % kw2;
  const int P = s & 7;
  frag_rowcol(tile, 2 * wi + k_local_of_pair(P), lane, reg_of_pair(P), s >> 3, tok, v);
}

// Value word w, code slot s -> (tok, ch).
__host__ __device__ inline void value_word_code(int w, int s, int bits, int& tok, int& ch) {
  int tile, k, lane, reg, half, row, col;
  lane = (w >> 2) & 31;
  if (bits == 2) {
    tile = w >> 7;
    half = s >> 3;
    const int P = s & 7;
    reg = reg_of_pair(P);
    k = 2 * (w & 3) + k_local_of_pair(P);
  } else {
    tile = w >> 8;
    k = 4 * ((w >> 7) & 1) + (w & 3);
    half = s >> 2;
    reg = reg_of_nibble(s & 3);
  }
  frag_rowcol(tile, k, lane, reg, half, row, col);
  ch = row;
  tok = col;
}

}  // namespace kvq
