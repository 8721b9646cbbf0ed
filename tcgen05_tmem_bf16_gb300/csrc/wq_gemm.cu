// wq_gemm.cu -- weight-only quantised GEMM with on-chip dequantisation,
// sm_103a: int4, FP8 (E4M3) and NVFP4 (E2M1) weights, bf16 activations.
//
// The kernel streams the packed weights and their scales into shared memory
// with TMA, dequantises them on-chip to bf16, and feeds them to the tensor
// cores; the bf16 weight matrix never exists in HBM ("Fusion Thinking",
// Pattern 3, Dequant + GEMM: load the quantised weights + scales directly,
// unpack, w = (q - 8) * s for int4, accumulate a . w; the same pattern names
// NVFP4 weight-only quantisation with BF16 activations).
//
// Weight formats (FMT):
//   int4   [K][N/2] bytes, two codes per byte along N (column 2j = high
//          nibble of byte j); w = bf16((q - 8) * s[k/G][n]), bf16 scales.
//   fp8    [K][N] E4M3 bytes; w = bf16(e4m3(q) * s[k/G][n]), bf16 scales.
//   nvfp4  [K][N/2] E2M1 codes packed like int4; w = e2m1(q) * e4m3(S[k/16][n])
//          (exact in bf16), E4M3 scale bytes [K/16][N]; the per-tensor
//          factor is the caller's alpha.
//
// GB300 design.  out^T = W~^T * A^T: the weights are the MMA's A operand
// (128 rows = output columns) and the few activation rows are its N.  The
// dequantised A operand is written straight into TENSOR MEMORY with
// tcgen05.st and consumed by tcgen05.mma from there, so the 2-byte weights
// never make a round trip through shared memory: per weight, shared memory
// carries only the half byte the TMA engine wrote and the transform threads
// read once.
//
// Tile: 512 output columns.  Transform thread t (TMEM lane t) owns output
// columns n0+4t .. n0+4t+3 of every k-row: packed bytes 2t and 2t+1 for the
// 4-bit formats (high nibble of byte 2t, low nibble of 2t, high of 2t+1, low
// of 2t+1), bytes 4t .. 4t+3 for FP8.
// Those four columns are four 128-lane A operands ("regions" 0..3), so each
// thread writes only its own TMEM lane, one shared-memory load per k-row
// feeds four weights, and the epilogue stores four adjacent outputs at once.
// One 64-deep K block = 16 MMAs (4 regions x 4 steps of 16).
//
// Eight transform warps form two groups; group g dequantises k-rows
// [32g, 32g+32) of every shared-memory stage into its own TMEM buffer, so
// one group fills while the MMAs drain the other.
//
// Dequantisation of an int4 code q, exact as the definition wants:
//   bits 0x4300 | q  is the bf16 value 128 + q;
//   (128 + q) - 136 = q - 8 exactly (small integers);
//   (q - 8) * s with one bf16 multiply = bf16_rne((q - 8) * s).
// For a k-row pair the two 16-bit loads are joined into X = row_k | row_k+1
// << 16; the four regions are then (X >> 4), X, (X >> 12), (X >> 8) masked
// with 0x000F000F -- each a bf16x2 pair (k, k+1) after OR-ing 0x43004300.
// The floating-point codes are moved bit-wise into a bf16 whose exponent
// field holds the code's exponent field: an E4M3 byte S.EEEE.MMM becomes the
// bf16 S.0000EEEE.MMM0000 = value * 2^-120 and an E2M1 code S.EE.M the bf16
// S.000000EE.M000000 = value * 2^-126 (the codes' subnormals land on bf16
// subnormals with the same factor).  One exact bf16 multiply by 2^120 or
// 2^126 restores the value, a second multiplies by the scale (exact for
// NVFP4: at most 6 significant bits; the one rounding for FP8).
//
// K is split across a thread-block cluster; the ranks exchange partial sums
// through shared memory (each rank gets the other ranks' partials of its own
// output rows by bulk copy, or loads them through distributed shared memory
// for the larger tile of M > 16), sum them in rank order and apply the
// ending once.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace gbf {

constexpr int kW4Threads = 384;                 // warps 0-3 roles, 4-11 transform/epilogue
constexpr int kW4Regions = 4;
constexpr uint32_t kBf16x2Pow120 = 0x7B807B80u;  // bf16x2 (2^120, 2^120)

template <int FMT, int MPAD>
struct W4Cfg {
  static constexpr int kRowBytes = FMT == kWqFp8 ? kW4BN : kW4BN / 2;  // weight bytes per k-row
  static constexpr int kQBytes = kBK * kRowBytes;                      // weight tile per stage
  static constexpr int kXBytes = MPAD * kBK * 2;                       // activations, SW128
  // int4 / fp8: one row of 512 bf16 group scales per stage (G % 64 == 0);
  // nvfp4: four rows (k-blocks of 16) of 512 E4M3 bytes.
  static constexpr int kScaleBytes = FMT == kWqNvfp4 ? 2048 : 1024;
  static constexpr int kStageBytes = kQBytes + kXBytes + kScaleBytes;
  static constexpr int kStages = FMT == kWqFp8 ? 3 : (MPAD <= 16 ? 5 : 4);
  static constexpr int kSmem = 1024 + kStages * kStageBytes + 256;
  static constexpr uint32_t kTmemCols = 256;
  // Tensor-memory pipeline between the transform warps and the MMAs.
  //
  // Accumulators: kSets copies of the four region accumulators, D(set e,
  // region r) at columns (4e + r) * MPAD.  With one set the two MMA issuers
  // split the regions (issuer i owns regions 2i and 2i+1, every K step);
  // with two sets issuer i owns set i and takes every other operand unit.
  // Either way every accumulator has exactly one writer, and the epilogue
  // adds the sets, set 0 first.
  //
  // Operand units: the dequantised weights of kUnitRows k-rows (all four
  // regions, kUnitRows / 2 columns each) are one hand-over from a transform
  // group to the MMAs.  The units of consecutive stages go round a ring of
  // kBufs tensor-memory buffers, so a transform group refills a buffer while
  // the MMAs still read the previous ones; a buffer is released when every
  // MMA that reads it has completed.
  static constexpr int kSets = 1;
  static constexpr int kUnitRows = 32;
  static constexpr int kIssuers = 2;
  static constexpr int kUnits = kBK / kUnitRows;        // units per stage (2 per group or 1)
  static constexpr int kUnitCols = 2 * kUnitRows;       // 4 regions x kUnitRows / 2 columns
  static constexpr uint32_t kColA = kSets * kW4Regions * MPAD;
  static constexpr int kBufs = (kTmemCols - kColA) / kUnitCols;
  static_assert(kBufs >= 2 && kBufs <= 8, "operand ring of two to eight buffers");
  static_assert(kColA + kBufs * kUnitCols <= kTmemCols, "TMEM budget");
  static_assert(kUnits % 2 == 0, "each transform group fills whole units");
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");
  static_assert(kStages * kStageBytes >= 128 * kW4Regions * MPAD * 4, "reduction buffer");
  static_assert(kSmem <= 115 * 1024, "two CTAs per SM");
  // Split-K exchange by pushing (see the kernel's epilogue): the partial
  // (MPAD rows of 128 lanes x 4 regions, fp32) plus the largest receive area
  // (S * ceil(MPAD / S) < MPAD + kMaxSplits rows) must fit in the stage
  // memory; otherwise the ranks pull through distributed shared memory.
  static constexpr int kRowPartBytes = 128 * kW4Regions * 4;
  static constexpr bool kPush = (2 * MPAD + kMaxSplits) * kRowPartBytes <= kStages * kStageBytes;
};

struct W4Args {
  int M, N, K;
  int num_kb;
  int splits;
  EpiParams ep;
  KernelCtl ctl;
};

// One k-row pair of this thread's two packed bytes -> the four dequantised
// bf16x2 pairs (regions 0..3).  x0, x1: the 16-bit loads of rows k and k+1
// (zero-extended).  In explicit PTX so that each step is one instruction:
// join (prmt), three shifts, four lop3 ((v & 0x000F000F) | 0x43004300 gives
// bf16 128+q in each half), and per pair one sub.rn.bf16x2 (-136, exact) and
// one mul.rn.bf16x2 (x s, the single rounding the definition asks for).
__device__ __forceinline__ void deq_rowpair(uint32_t x0, uint32_t x1, uint32_t c136,
                                            uint32_t s0, uint32_t s1, uint32_t s2, uint32_t s3,
                                            uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                            uint32_t& o3) {
  asm("{\n\t"
      ".reg .b32 x, t0, t1, t2, t3;\n\t"
      "prmt.b32 x, %4, %5, 0x5410;\n\t"
      "shr.b32 t0, x, 4;\n\t"
      "shr.b32 t2, x, 12;\n\t"
      "shr.b32 t3, x, 8;\n\t"
      "lop3.b32 t0, t0, 0x000F000F, 0x43004300, 0xEA;\n\t"
      "lop3.b32 t1, x, 0x000F000F, 0x43004300, 0xEA;\n\t"
      "lop3.b32 t2, t2, 0x000F000F, 0x43004300, 0xEA;\n\t"
      "lop3.b32 t3, t3, 0x000F000F, 0x43004300, 0xEA;\n\t"
      "sub.rn.bf16x2 t0, t0, %6;\n\t"
      "sub.rn.bf16x2 t1, t1, %6;\n\t"
      "sub.rn.bf16x2 t2, t2, %6;\n\t"
      "sub.rn.bf16x2 t3, t3, %6;\n\t"
      "mul.rn.bf16x2 %0, t0, %7;\n\t"
      "mul.rn.bf16x2 %1, t1, %8;\n\t"
      "mul.rn.bf16x2 %2, t2, %9;\n\t"
      "mul.rn.bf16x2 %3, t3, %10;\n\t"
      "}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(x0), "r"(x1), "r"(c136), "r"(s0), "r"(s1), "r"(s2), "r"(s3));
}

// The same with one fused multiply-add per bf16x2 pair, for scales with
// |s| < 2^-5.  A bf16 bit pattern p < 0x100 (exponent field 0 or 1) has the
// value p * 2^-133 exactly, so a nibble masked in place is already a bf16
// multiple of q: bits 0-3 give q * 2^-133, bits 4-7 give q * 2^-129.  With
// sp = s * 2^133 or s * 2^129 (exact: no overflow for such s) and c = -8 s
// (exact), fma(nibble, sp, c) = q*s - 8*s computed exactly and rounded once,
// i.e. bf16_rne((q - 8) * s) as the definition asks.  Regions 1 and 0 (low
// and high nibble of byte 2t) are masked in place, regions 3 and 2 after
// one shift by 8 (bits 8-15 of each half; the high half's upper byte that
// the shift brings into the low half is masked off).  10 instructions per
// k-row pair instead of 16.  sp0, sp2: s * 2^129; sp1, sp3: s * 2^133.
__device__ __forceinline__ void deq_rowpair_fma(uint32_t x0, uint32_t x1, uint32_t sp0,
                                                uint32_t sp1, uint32_t sp2, uint32_t sp3,
                                                uint32_t c0, uint32_t c1, uint32_t c2,
                                                uint32_t c3, uint32_t& o0, uint32_t& o1,
                                                uint32_t& o2, uint32_t& o3) {
  asm("{\n\t"
      ".reg .b32 x, y, t0, t1, t2, t3;\n\t"
      "prmt.b32 x, %4, %5, 0x5410;\n\t"
      "shr.b32 y, x, 8;\n\t"
      "and.b32 t0, x, 0x00F000F0;\n\t"
      "and.b32 t1, x, 0x000F000F;\n\t"
      "and.b32 t2, y, 0x00F000F0;\n\t"
      "and.b32 t3, y, 0x000F000F;\n\t"
      "fma.rn.bf16x2 %0, t0, %6, %10;\n\t"
      "fma.rn.bf16x2 %1, t1, %7, %11;\n\t"
      "fma.rn.bf16x2 %2, t2, %8, %12;\n\t"
      "fma.rn.bf16x2 %3, t3, %9, %13;\n\t"
      "}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(x0), "r"(x1), "r"(sp0), "r"(sp1), "r"(sp2), "r"(sp3), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3));
}

// bf16x2 a * b (round to nearest even).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// |value| of a bf16x2 (s, s) pair below the bf16 `limit_bits` (NaN and
// infinity are not).
__device__ __forceinline__ bool bf16_abs_below(uint32_t pair, uint32_t limit_bits) {
  return (pair & 0x7FFFu) < limit_bits;
}

// FP8 k-row pair: x0, x1 = the 32-bit loads (bytes = columns 4t..4t+3) of
// rows k and k+1.  Region r: prmt puts byte r of each row into bytes 1 and 3
// (the high byte of each half), the magnitude bits move down by 4 into the
// bf16 exponent/mantissa fields, the sign bit stays at bit 15 / 31; then
// x 2^120 (exact) and x s (the one rounding).
__device__ __forceinline__ void deq_fp8_rowpair(uint32_t x0, uint32_t x1, uint32_t s0,
                                                uint32_t s1, uint32_t s2, uint32_t s3,
                                                uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                                uint32_t& o3) {
  asm("{\n\t"
      ".reg .b32 y, u;\n\t"
      "prmt.b32 y, %4, %5, 0x4400;\n\t"
      "and.b32 u, y, 0x7F007F00;\n\t"
      "shr.b32 u, u, 4;\n\t"
      "lop3.b32 u, u, y, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 u, u, %10;\n\t"
      "mul.rn.bf16x2 %0, u, %6;\n\t"
      "prmt.b32 y, %4, %5, 0x5511;\n\t"
      "and.b32 u, y, 0x7F007F00;\n\t"
      "shr.b32 u, u, 4;\n\t"
      "lop3.b32 u, u, y, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 u, u, %10;\n\t"
      "mul.rn.bf16x2 %1, u, %7;\n\t"
      "prmt.b32 y, %4, %5, 0x6622;\n\t"
      "and.b32 u, y, 0x7F007F00;\n\t"
      "shr.b32 u, u, 4;\n\t"
      "lop3.b32 u, u, y, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 u, u, %10;\n\t"
      "mul.rn.bf16x2 %2, u, %8;\n\t"
      "prmt.b32 y, %4, %5, 0x7733;\n\t"
      "and.b32 u, y, 0x7F007F00;\n\t"
      "shr.b32 u, u, 4;\n\t"
      "lop3.b32 u, u, y, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 u, u, %10;\n\t"
      "mul.rn.bf16x2 %3, u, %9;\n\t"
      "}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(x0), "r"(x1), "r"(s0), "r"(s1), "r"(s2), "r"(s3), "r"(kBf16x2Pow120));
}

// The same with the two multiplies fused, for scales with |s| < 2^8: with
// sp = s * 2^120 (exact), code * 2^-120 * sp is the exact product e4m3 * s,
// rounded once.  20 instructions per k-row pair instead of 24.
__device__ __forceinline__ void deq_fp8_rowpair_fused(uint32_t x0, uint32_t x1, uint32_t sp0,
                                                      uint32_t sp1, uint32_t sp2, uint32_t sp3,
                                                      uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                                      uint32_t& o3) {
  asm("{\n\t"
      ".reg .b32 y, u;\n\t"
      "prmt.b32 y, %4, %5, 0x4400;\n\t"
      "and.b32 u, y, 0x7F007F00;\n\t"
      "shr.b32 u, u, 4;\n\t"
      "lop3.b32 u, u, y, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 %0, u, %6;\n\t"
      "prmt.b32 y, %4, %5, 0x5511;\n\t"
      "and.b32 u, y, 0x7F007F00;\n\t"
      "shr.b32 u, u, 4;\n\t"
      "lop3.b32 u, u, y, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 %1, u, %7;\n\t"
      "prmt.b32 y, %4, %5, 0x6622;\n\t"
      "and.b32 u, y, 0x7F007F00;\n\t"
      "shr.b32 u, u, 4;\n\t"
      "lop3.b32 u, u, y, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 %2, u, %8;\n\t"
      "prmt.b32 y, %4, %5, 0x7733;\n\t"
      "and.b32 u, y, 0x7F007F00;\n\t"
      "shr.b32 u, u, 4;\n\t"
      "lop3.b32 u, u, y, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 %3, u, %9;\n\t"
      "}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(x0), "r"(x1), "r"(sp0), "r"(sp1), "r"(sp2), "r"(sp3));
}

// Four E4M3 scale bytes (columns 4t..4t+3) -> four bf16x2 (s, s) pairs, exact.
__device__ __forceinline__ void e4m3x4_to_bf16x2_dup(uint32_t b, uint32_t& s0, uint32_t& s1,
                                                     uint32_t& s2, uint32_t& s3) {
  asm("{\n\t"
      ".reg .b32 y, u;\n\t"
      "prmt.b32 y, %4, %4, 0x0000;\n\t"
      "and.b32 u, y, 0x7F007F00;\n\t"
      "shr.b32 u, u, 4;\n\t"
      "lop3.b32 u, u, y, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 %0, u, %5;\n\t"
      "prmt.b32 y, %4, %4, 0x1111;\n\t"
      "and.b32 u, y, 0x7F007F00;\n\t"
      "shr.b32 u, u, 4;\n\t"
      "lop3.b32 u, u, y, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 %1, u, %5;\n\t"
      "prmt.b32 y, %4, %4, 0x2222;\n\t"
      "and.b32 u, y, 0x7F007F00;\n\t"
      "shr.b32 u, u, 4;\n\t"
      "lop3.b32 u, u, y, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 %2, u, %5;\n\t"
      "prmt.b32 y, %4, %4, 0x3333;\n\t"
      "and.b32 u, y, 0x7F007F00;\n\t"
      "shr.b32 u, u, 4;\n\t"
      "lop3.b32 u, u, y, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 %3, u, %5;\n\t"
      "}"
      : "=r"(s0), "=r"(s1), "=r"(s2), "=r"(s3)
      : "r"(b), "r"(kBf16x2Pow120));
}

// NVFP4 k-row pairs: x0, x1 = the 16-bit loads of rows k and k+1 (packed
// bytes 2t, 2t+1), joined into X.  Region r's nibble sits at bits 4/0/12/8 of
// each half; its magnitude bits (EE.M) move to bf16 bits 6..8 and its sign bit
// to bit 15, which reads as e2m1 * 2^-126 (the code 0.5 as a bf16 subnormal).
//
// NVFP4 operand scaled by an exact power of two: with sp = s * 2^107 (exact:
// s <= 448), one multiply gives e2m1 * s * 2^-19 instead of e2m1 * s (the code
// read as bf16 is e2m1 * 2^-126; the product has at most 6 significant bits
// and lies in [2^-29, 2^-7.6], so it is exact and a normal bf16).  The MMA
// then accumulates the product scaled by 2^-19, which fp32 does exactly as
// it would the unscaled one (a power-of-two factor commutes with every
// rounding while nothing underflows), and the ending multiplies by 2^19
// through alpha.  5 instructions per bf16 pair instead of 6.
constexpr float kNvfp4OperandScale = 524288.0f;  // 2^19, restored in the ending
constexpr uint32_t kBf16x2Pow107 = 0x75007500u;  // bf16x2 (2^107, 2^107)

__device__ __forceinline__ void deq_fp4_rowpair_scaled(uint32_t x0, uint32_t x1, uint32_t sp0,
                                                       uint32_t sp1, uint32_t sp2, uint32_t sp3,
                                                       uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                                       uint32_t& o3) {
  asm("{\n\t"
      ".reg .b32 x, a, b;\n\t"
      "prmt.b32 x, %4, %5, 0x5410;\n\t"
      "shl.b32 a, x, 2;\n\t"
      "shl.b32 b, x, 8;\n\t"
      "and.b32 a, a, 0x01C001C0;\n\t"
      "lop3.b32 a, a, b, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 %0, a, %6;\n\t"
      "shl.b32 a, x, 6;\n\t"
      "shl.b32 b, x, 12;\n\t"
      "and.b32 a, a, 0x01C001C0;\n\t"
      "lop3.b32 a, a, b, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 %1, a, %7;\n\t"
      "shr.b32 a, x, 6;\n\t"
      "and.b32 a, a, 0x01C001C0;\n\t"
      "lop3.b32 a, a, x, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 %2, a, %8;\n\t"
      "shr.b32 a, x, 2;\n\t"
      "shl.b32 b, x, 4;\n\t"
      "and.b32 a, a, 0x01C001C0;\n\t"
      "lop3.b32 a, a, b, 0x80008000, 0xF8;\n\t"
      "mul.rn.bf16x2 %3, a, %9;\n\t"
      "}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(x0), "r"(x1), "r"(sp0), "r"(sp1), "r"(sp2), "r"(sp3));
}

// Epilogue of output columns n..n+3 for 8 rows m0..m0+7: operand loads
// first (independent, overlapping), then the math and 8-byte stores.
template <int ACT>
__device__ __forceinline__ void epi_quad8(const float (&v)[kW4Regions][8], int64_t m0, int n,
                                          int M, int N, const EpiParams& e) {
  if (n >= N) return;
  float b[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (e.bias) {
    const uint2 bb = *reinterpret_cast<const uint2*>(e.bias + n);
    b[0] = bf16lo(bb.x); b[1] = bf16hi(bb.x); b[2] = bf16lo(bb.y); b[3] = bf16hi(bb.y);
  }
  const float beta = e.C ? e.beta : 0.0f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // two halves of 4 rows keep the register count low
    uint2 c[4], r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t m = m0 + 4 * h + j;
      const bool ok = m < M;
      const int64_t off = m * N + n;
      c[j] = (ok && e.C) ? *reinterpret_cast<const uint2*>(e.C + off) : make_uint2(0, 0);
      r[j] = (ok && e.residual) ? *reinterpret_cast<const uint2*>(e.residual + off)
                                : make_uint2(0, 0);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t m = m0 + 4 * h + j;
      if (m >= M) break;
      const float cc[4] = {bf16lo(c[j].x), bf16hi(c[j].x), bf16lo(c[j].y), bf16hi(c[j].y)};
      const float rr[4] = {bf16lo(r[j].x), bf16hi(r[j].x), bf16lo(r[j].y), bf16hi(r[j].y)};
      float x[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        x[q] = act_apply<ACT>(fmaf(beta, cc[q], e.alpha * v[q][4 * h + j]) + b[q]) + rr[q];
      *reinterpret_cast<uint2*>(e.out + m * N + n) =
          make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
    }
  }
}

// Epilogue of output columns n..n+3 of one row m.
template <int ACT>
__device__ __forceinline__ void epi_quad1(const float4& v, int64_t m, int n, int M, int N,
                                          const EpiParams& e) {
  if (n >= N || m >= M) return;
  const int64_t off = m * N + n;
  const uint2 c = e.C ? *reinterpret_cast<const uint2*>(e.C + off) : make_uint2(0, 0);
  const uint2 r = e.residual ? *reinterpret_cast<const uint2*>(e.residual + off)
                             : make_uint2(0, 0);
  float b[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (e.bias) {
    const uint2 bb = *reinterpret_cast<const uint2*>(e.bias + n);
    b[0] = bf16lo(bb.x); b[1] = bf16hi(bb.x); b[2] = bf16lo(bb.y); b[3] = bf16hi(bb.y);
  }
  const float beta = e.C ? e.beta : 0.0f;
  const float acc[4] = {v.x, v.y, v.z, v.w};
  const float cc[4] = {bf16lo(c.x), bf16hi(c.x), bf16lo(c.y), bf16hi(c.y)};
  const float rr[4] = {bf16lo(r.x), bf16hi(r.x), bf16lo(r.y), bf16hi(r.y)};
  float x[4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    x[q] = act_apply<ACT>(fmaf(beta, cc[q], e.alpha * acc[q]) + b[q]) + rr[q];
  *reinterpret_cast<uint2*>(e.out + off) =
      make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
}

template <int FMT, int MPAD>
__global__ void __launch_bounds__(kW4Threads, 2)
    wq_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmS, const W4Args a, int group) {
  using Cfg = W4Cfg<FMT, MPAD>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment by pointer arithmetic on the shared array (keeps the
  // shared address space for the compiler).
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kStages * Cfg::kStageBytes);
  uint64_t* empty = full + Cfg::kStages;
  uint64_t* afull = empty + Cfg::kStages;  // [kBufs]: operand buffer written
  uint64_t* aempty = afull + Cfg::kBufs;   // [kBufs]: operand buffer read by the MMAs
  uint64_t* dfull = aempty + Cfg::kBufs;
  uint64_t* done = dfull + 1;
  uint64_t* recvb = done + 1;  // split-K partials pushed here by the other ranks
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(recvb + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = a.splits;
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0;
  const int nb = blockIdx.y;
  const int mb = blockIdx.z;
  const int kb0 = static_cast<int>((static_cast<int64_t>(rank) * a.num_kb) / S);
  const int kb1 = static_cast<int>((static_cast<int64_t>(rank + 1) * a.num_kb) / S);

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 8 + Cfg::kIssuers);  // 8 transform warps + the MMA commits
    }
    for (int i = 0; i < Cfg::kBufs; ++i) {
      mbar_init(&afull[i], 4);                              // the writing group's 4 warps
      mbar_init(&aempty[i], Cfg::kSets == 1 ? 2 : 1);       // the commits of its readers
    }
    mbar_init(dfull, Cfg::kIssuers);
    mbar_init(done, Cfg::kIssuers);
    if (Cfg::kPush && S > 1) {
      // expects the other S - 1 ranks' copies of this rank's rows
      const int r = static_cast<int>(rank);
      const int nrow = ((r + 1) * MPAD) / S - (r * MPAD) / S;
      mbar_init(recvb, 1);
      mbar_arrive_expect_tx(recvb, static_cast<uint32_t>((S - 1) * nrow * Cfg::kRowPartBytes));
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmS);
  }
  if (warp == 2) {
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const WaitCtl ctl{a.ctl.err, a.ctl.timeout_ns, abort_flag, prof_slots(a.ctl.prof)};
  const long long t_start = clock64();
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t stream_policy = policy_evict_first();
      uint32_t fills[Cfg::kStages];
#pragma unroll
      for (int i = 0; i < Cfg::kStages; ++i) fills[i] = 0;
      // weight codes and scales of k block kb into stage s (read-only inputs)
      auto load_w = [&](int s, int kb) {
        uint8_t* sq = stages + s * Cfg::kStageBytes;
        uint8_t* ss = sq + Cfg::kQBytes + Cfg::kXBytes;
        // scale rows: one group row (int4, fp8) or four 16-deep blocks (nvfp4)
        const int srow = FMT == kWqNvfp4 ? kb * (kBK / 16) : (kb * kBK) / group;
        // the weight tile in boxes of 256 bytes x 64 k-rows
#pragma unroll
        for (int h = 0; h < Cfg::kRowBytes / 256; ++h)
          tma_load_2d_hint(sq + h * (kBK * 256), &tmQ, &full[s], nb * Cfg::kRowBytes + 256 * h,
                           kb * kBK, stream_policy);
        tma_load_2d(ss, &tmS, &full[s], nb * kW4BN, srow);
        tma_load_2d(ss + Cfg::kScaleBytes / 2, &tmS, &full[s], nb * kW4BN + 256, srow);
      };
      auto load_x = [&](int s, int kb) {
        tma_load_2d(stages + s * Cfg::kStageBytes + Cfg::kQBytes, &tmA, &full[s], kb * kBK,
                    mb * MPAD);
      };
      // Nothing is read before the previous kernel in the stream has
      // completed: any input, weights included, may be its output.
      griddep_wait();
      int s = 0;
      uint32_t ph = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_bar(&empty[s], ph ^ 1, ctl, kSiteProducerEmpty)) break;
        mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
        load_w(s, kb);
        load_x(s, kb);
        fills[s]++;
        if (++s == Cfg::kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      for (int i = 0; i < Cfg::kStages; ++i)
        if (fills[i]) wait_bar(&full[i], (fills[i] - 1) & 1, ctl, kSiteDrain, false);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    // The operand units of the CTA's K range in order h = 0, 1, ...; unit h
    // sits in buffer h % kBufs.  One set: both issuers read every unit, each
    // into its own two regions.  Two sets: issuer i reads units h % 2 == i,
    // all four regions, into set i.
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, MPAD, false, false);
      constexpr int kSteps = Cfg::kUnitRows / 16;   // 16-deep K steps per unit
      constexpr int kRegionCols = Cfg::kUnitRows / 2;
      const int issuer = warp == 1 ? 0 : 1;
      const int r0 = Cfg::kSets == 1 ? 2 * issuer : 0;
      const int r1 = Cfg::kSets == 1 ? r0 + 2 : kW4Regions;
      const uint32_t dset = tmem_base + (Cfg::kSets == 1 ? 0 : issuer) * kW4Regions * MPAD;
      int s = 0;
      uint32_t ph = 0;
      int b = 0;          // buffer of unit h
      uint32_t bph = 0;   // parity of unit h's use of that buffer
      int h = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1 && ok; ++kb) {
        if (!wait_bar(&full[s], ph, ctl, kSiteMmaFull)) {
          ok = false;
          break;
        }
        const uint32_t x0 = smem_u32(stages + s * Cfg::kStageBytes + Cfg::kQBytes);
        for (int uu = 0; uu < Cfg::kUnits; ++uu, ++h) {
          if (Cfg::kSets == 1 || (h & 1) == issuer) {
            if (!wait_bar(&afull[b], bph, ctl, kSiteMmaOperand)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t abuf = tmem_base + Cfg::kColA + Cfg::kUnitCols * b;
#pragma unroll
            for (int k = 0; k < kSteps; ++k) {
              // activation rows of k-rows [uu * kUnitRows + 16 k, +16) of the stage
              const uint64_t bd = sdesc_sw128(x0 + (uu * kSteps + k) * 32, 16, 1024);
              // the first K step into an accumulator overwrites it
              const uint32_t accum = (h >= Cfg::kSets || k > 0) ? 1u : 0u;
#pragma unroll
              for (int r = r0; r < r1; ++r)
                mma_ts(dset + r * MPAD, abuf + kRegionCols * r + 8 * k, bd, idesc, accum);
            }
            mma_commit(&aempty[b]);
          }
          if (++b == Cfg::kBufs) {
            b = 0;
            bph ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&empty[s]);
        if (++s == Cfg::kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (ok && !a.ctl.inject) mma_commit(dfull);
      mma_commit(done);
      wait_bar(done, 0, ctl, kSiteDrain, false);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ dequantise into TMEM
    const int g = (warp - 4) >> 2;          // group: k-rows [32g, 32g + 32) of each stage
    const int q = warp & 3;                 // TMEM lane quarter
    const int t = q * 32 + lane;            // TMEM lane = owner of packed bytes 2t, 2t+1
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t lane_base = tmem_base + lane_off + Cfg::kColA;
    constexpr int kHalvesPerUnit = Cfg::kUnitRows / 16;  // 16-row halves of a unit
    constexpr int kRegionCols = Cfg::kUnitRows / 2;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    // Each 16-row half of the group's 32 rows is dequantised in registers
    // first; only then is the unit's buffer waited for, so that this work
    // overlaps the MMAs still reading the buffer's previous unit.
    for (int kb = kb0; kb < kb1 && ok; ++kb) {
      if (!wait_bar(&full[s], ph, ctl, kSiteXformFull)) break;
      const int j = kb - kb0;
      const uint8_t* sq = stages + s * Cfg::kStageBytes;
      const uint8_t* ssc = sq + Cfg::kQBytes + Cfg::kXBytes;
      int cur = 0;         // buffer of the unit being filled
      uint32_t ubuf = 0;   // its TMEM address in this warp's lane quarter
      // wait until the unit holding half `hh` of this group's rows has a free buffer
      auto acquire = [&](int hh) -> bool {
        const int h = Cfg::kUnits * j + (Cfg::kUnits / 2) * g + hh / kHalvesPerUnit;
        cur = h % Cfg::kBufs;
        const uint32_t use = static_cast<uint32_t>(h / Cfg::kBufs);
        if (!wait_bar(&aempty[cur], (use & 1) ^ 1, ctl, kSiteXformEmpty)) return false;
        tc_fence_after();
        ubuf = lane_base + Cfg::kUnitCols * cur;
        return true;
      };
      // store half `hh` (eight bf16x2 k-row pairs of each region)
      auto put = [&](int hh, const uint32_t (&o0)[8], const uint32_t (&o1)[8],
                     const uint32_t (&o2)[8], const uint32_t (&o3)[8]) {
        const uint32_t c = 8 * (hh % kHalvesPerUnit);
        tmem_st8(ubuf + c, o0);
        tmem_st8(ubuf + kRegionCols + c, o1);
        tmem_st8(ubuf + 2 * kRegionCols + c, o2);
        tmem_st8(ubuf + 3 * kRegionCols + c, o3);
        if (hh % kHalvesPerUnit == kHalvesPerUnit - 1) {  // the unit is complete
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&afull[cur]);
        }
      };
      // one 16-row half: dequantise its 8 k-row pairs with `deq`
      // (x0, x1 -> four bf16x2), then hand it to the unit's buffer
      auto half = [&](int hh, const uint8_t* rows, int row_bytes, auto deq) -> bool {
        uint32_t o0[8], o1[8], o2[8], o3[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int row = 16 * hh + 2 * p;
          deq(rows + row * row_bytes, rows + (row + 1) * row_bytes, o0[p], o1[p], o2[p], o3[p]);
        }
        if (hh % kHalvesPerUnit == 0 && !acquire(hh)) return false;
        put(hh, o0, o1, o2, o3);
        return true;
      };
      if constexpr (FMT == kWqFp8) {
        // bytes 4t..4t+3 of each k-row: box half t/64, word t%64
        const uint2 sc = *reinterpret_cast<const uint2*>(ssc + 8 * t);
        const uint32_t s0 = __byte_perm(sc.x, 0, 0x1010);
        const uint32_t s1 = __byte_perm(sc.x, 0, 0x3232);
        const uint32_t s2 = __byte_perm(sc.y, 0, 0x1010);
        const uint32_t s3 = __byte_perm(sc.y, 0, 0x3232);
        const uint8_t* rows = sq + (t >> 6) * (kBK * 256) + (32 * g) * 256 + 4 * (t & 63);
        // |s| < 2^8 on every lane: one multiply by s * 2^120 per pair
        constexpr uint32_t kLimit = 0x4380u;  // bf16 2^8
        if (__all_sync(0xffffffffu, bf16_abs_below(s0, kLimit) && bf16_abs_below(s1, kLimit) &&
                                        bf16_abs_below(s2, kLimit) && bf16_abs_below(s3, kLimit))) {
          const uint32_t p0 = bf16x2_mul(s0, kBf16x2Pow120), p1 = bf16x2_mul(s1, kBf16x2Pow120);
          const uint32_t p2 = bf16x2_mul(s2, kBf16x2Pow120), p3 = bf16x2_mul(s3, kBf16x2Pow120);
          auto deq = [=](const uint8_t* r0, const uint8_t* r1, uint32_t& a0, uint32_t& a1,
                         uint32_t& a2, uint32_t& a3) {
            deq_fp8_rowpair_fused(*reinterpret_cast<const uint32_t*>(r0),
                                  *reinterpret_cast<const uint32_t*>(r1), p0, p1, p2, p3, a0, a1,
                                  a2, a3);
          };
#pragma unroll
          for (int hh = 0; hh < 2 && ok; ++hh) ok = half(hh, rows, 256, deq);
        } else {
          auto deq = [=](const uint8_t* r0, const uint8_t* r1, uint32_t& a0, uint32_t& a1,
                         uint32_t& a2, uint32_t& a3) {
            deq_fp8_rowpair(*reinterpret_cast<const uint32_t*>(r0),
                            *reinterpret_cast<const uint32_t*>(r1), s0, s1, s2, s3, a0, a1, a2,
                            a3);
          };
#pragma unroll
          for (int hh = 0; hh < 2 && ok; ++hh) ok = half(hh, rows, 256, deq);
        }
      } else if constexpr (FMT == kWqInt4) {
        const uint8_t* rows = sq + (32 * g) * Cfg::kRowBytes + 2 * t;
        const uint2 sc = *reinterpret_cast<const uint2*>(ssc + 8 * t);
        const uint32_t s0 = __byte_perm(sc.x, 0, 0x1010);  // bf16x2 (s, s), column 4t
        const uint32_t s1 = __byte_perm(sc.x, 0, 0x3232);  // column 4t+1
        const uint32_t s2 = __byte_perm(sc.y, 0, 0x1010);  // column 4t+2
        const uint32_t s3 = __byte_perm(sc.y, 0, 0x3232);  // column 4t+3
        // regions: 0 = high nibble of byte 2t, 1 = low of 2t, 2 = high of 2t+1,
        // 3 = low of 2t+1
        constexpr uint32_t kLimit = 0x3D00u;  // bf16 2^-5
        if (__all_sync(0xffffffffu, bf16_abs_below(s0, kLimit) && bf16_abs_below(s1, kLimit) &&
                                        bf16_abs_below(s2, kLimit) && bf16_abs_below(s3, kLimit))) {
          // s * 2^129 for the high nibbles, s * 2^133 for the low ones
          // (products of exact power-of-two factors), and -8 s (exact)
          constexpr uint32_t kPow126 = 0x7E807E80u, kPow3 = 0x41004100u, kPow7 = 0x43004300u;
          constexpr uint32_t kMinus8 = 0xC100C100u;
          const uint32_t p0 = bf16x2_mul(bf16x2_mul(s0, kPow126), kPow3);
          const uint32_t p1 = bf16x2_mul(bf16x2_mul(s1, kPow126), kPow7);
          const uint32_t p2 = bf16x2_mul(bf16x2_mul(s2, kPow126), kPow3);
          const uint32_t p3 = bf16x2_mul(bf16x2_mul(s3, kPow126), kPow7);
          const uint32_t c0 = bf16x2_mul(s0, kMinus8), c1 = bf16x2_mul(s1, kMinus8);
          const uint32_t c2 = bf16x2_mul(s2, kMinus8), c3 = bf16x2_mul(s3, kMinus8);
          auto deq = [=](const uint8_t* r0, const uint8_t* r1, uint32_t& a0, uint32_t& a1,
                         uint32_t& a2, uint32_t& a3) {
            deq_rowpair_fma(*reinterpret_cast<const uint16_t*>(r0),
                            *reinterpret_cast<const uint16_t*>(r1), p0, p1, p2, p3, c0, c1, c2,
                            c3, a0, a1, a2, a3);
          };
#pragma unroll
          for (int hh = 0; hh < 2 && ok; ++hh) ok = half(hh, rows, Cfg::kRowBytes, deq);
        } else {
          auto deq = [=](const uint8_t* r0, const uint8_t* r1, uint32_t& a0, uint32_t& a1,
                         uint32_t& a2, uint32_t& a3) {
            deq_rowpair(*reinterpret_cast<const uint16_t*>(r0),
                        *reinterpret_cast<const uint16_t*>(r1), 0x43084308u, s0, s1, s2, s3, a0,
                        a1, a2, a3);
          };
#pragma unroll
          for (int hh = 0; hh < 2 && ok; ++hh) ok = half(hh, rows, Cfg::kRowBytes, deq);
        }
      } else {
        const uint8_t* rows = sq + (32 * g) * Cfg::kRowBytes + 2 * t;
#pragma unroll
        for (int hh = 0; hh < 2 && ok; ++hh) {
          // the E4M3 block scale of k-rows [32g + 16hh, +16): block row 2g + hh
          uint32_t s0, s1, s2, s3;
          const uint32_t sb = *reinterpret_cast<const uint32_t*>(
              ssc + (t >> 6) * 1024 + (2 * g + hh) * 256 + 4 * (t & 63));
          e4m3x4_to_bf16x2_dup(sb, s0, s1, s2, s3);
          // s * 2^107 (exact), for the operand scaled by 2^-19
          const uint32_t p0 = bf16x2_mul(s0, kBf16x2Pow107), p1 = bf16x2_mul(s1, kBf16x2Pow107);
          const uint32_t p2 = bf16x2_mul(s2, kBf16x2Pow107), p3 = bf16x2_mul(s3, kBf16x2Pow107);
          auto deq = [=](const uint8_t* r0, const uint8_t* r1, uint32_t& a0, uint32_t& a1,
                         uint32_t& a2, uint32_t& a3) {
            deq_fp4_rowpair_scaled(*reinterpret_cast<const uint16_t*>(r0),
                                   *reinterpret_cast<const uint16_t*>(r1), p0, p1, p2, p3, a0,
                                   a1, a2, a3);
          };
          ok = half(hh, rows, Cfg::kRowBytes, deq);
        }
      }
      if (!ok) break;
      __syncwarp();  // every lane's shared-memory reads of the stage are done
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == Cfg::kStages) {
        s = 0;
        ph ^= 1;
      }
    }
  }

  // ---- epilogue: cluster reduction of the partial sums, then the ending.
  // Every rank parks its partial in its own shared memory.  Push exchange
  // (when it fits): the output rows are shared out among the ranks in
  // contiguous ranges, each rank copies every other rank's rows to that rank
  // with one bulk copy, and each rank sums its own rows over ranks 0..S-1 in
  // that order (deterministic) from local shared memory.  Otherwise 8-row
  // chunks go to the (rank, group) workers round-robin and are summed over
  // ranks 0..S-1 in that order through distributed shared memory.
  const bool epi = warp >= 4;
  if (epi) griddep_wait();  // the ending reads C, bias, residual and writes out
  const int g = (warp - 4) >> 2;
  const int q = warp & 3;
  const int tid = q * 32 + lane;
  const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  float4* red = reinterpret_cast<float4*>(stages);
  constexpr int kChunks = MPAD / 8;
  bool have = false;
  bool pushed = false;
  if constexpr (Cfg::kPush) {
    if (S > 1) {
      pushed = true;
      const int r = static_cast<int>(rank);
      const int ra = (r * MPAD) / S;  // this rank's rows [ra, ra + nrow)
      const int nrow = ((r + 1) * MPAD) / S - ra;
      uint8_t* recv = stages + MPAD * Cfg::kRowPartBytes;  // [sender][row][lane] float4
      if (epi) {
        have = wait_bar(dfull, 0, ctl, kSiteEpiAccFull);
        tc_fence_after();
        // park red[m * 128 + lane] = the lane's four columns of row m; group g
        // takes the 8-row chunks c = g, g + 2, ..., one region at a time
        float* redf = reinterpret_cast<float*>(stages);
#pragma unroll 1
        for (int c = g; c < kChunks; c += 2) {
#pragma unroll 1
          for (int rg = 0; rg < kW4Regions; ++rg) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = 0.0f;
#pragma unroll
            for (int e = 0; e < Cfg::kSets; ++e) {
              uint32_t u[8];
              tmem_ld8(tb + (e * kW4Regions + rg) * MPAD + c * 8, u);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] += __uint_as_float(u[j]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) redf[((c * 8 + j) * 128 + tid) * 4 + rg] = v[j];
          }
        }
        fence_proxy_async_smem();  // the bulk copies read what these threads wrote
      }
      cluster_sync_all();  // every rank parked, every receive barrier armed
      if (threadIdx.x == 128) {
        for (int i = 1; i < S; ++i) {
          const int p = (r + i) % S;
          const int pa = (p * MPAD) / S;
          const int pn = ((p + 1) * MPAD) / S - pa;
          if (pn > 0)
            bulk_copy_to_peer(
                mapa_shared(smem_u32(recv + r * pn * Cfg::kRowPartBytes), static_cast<uint32_t>(p)),
                smem_u32(stages + pa * Cfg::kRowPartBytes),
                static_cast<uint32_t>(pn * Cfg::kRowPartBytes),
                mapa_shared(smem_u32(recvb), static_cast<uint32_t>(p)));
        }
      }
      if (epi && nrow > 0) {
        // Not cut short by the abort flag: every peer issues its copies after
        // the cluster barrier above whatever its state, so this wait ends
        // (bounded by the timeout) and the final barrier then follows them.
        wait_bar(recvb, 0, ctl, kSiteEpiAccFull, /*honor_abort=*/false);
        const float4* in = reinterpret_cast<const float4*>(recv);
        const int n = nb * kW4BN + 4 * tid;
#pragma unroll 1
        for (int i = g; i < nrow; i += 2) {
          float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          for (int p = 0; p < S; ++p) {
            const float4 f = p == r ? red[(ra + i) * 128 + tid] : in[(p * nrow + i) * 128 + tid];
            if (p == 0) {
              t = f;
            } else {
              t.x += f.x;
              t.y += f.y;
              t.z += f.z;
              t.w += f.w;
            }
          }
          const int64_t row = static_cast<int64_t>(mb) * MPAD + ra + i;
          switch (a.ep.act) {
            case kActRelu: epi_quad1<kActRelu>(t, row, n, a.M, a.N, a.ep); break;
            case kActSilu: epi_quad1<kActSilu>(t, row, n, a.M, a.N, a.ep); break;
            case kActGeluTanh: epi_quad1<kActGeluTanh>(t, row, n, a.M, a.N, a.ep); break;
            default: epi_quad1<kActIdentity>(t, row, n, a.M, a.N, a.ep); break;
          }
        }
      }
      // No rank leaves while copies from or into its shared memory may be in
      // flight: every copy has completed on its receiver's barrier, which the
      // receiver waited for before arriving.  The arrival is relaxed, so it
      // does not first wait for this thread's stores of the ending.
      cluster_sync_relaxed_arrive();
    }
  }
  if (!pushed) {
  if (epi) {
    have = wait_bar(dfull, 0, ctl, kSiteEpiAccFull);
    tc_fence_after();
    if (!Cfg::kPush && S > 1 && g == 0) {  // (with the push exchange: S = 1 here)
#pragma unroll 1
      for (int r = 0; r < kW4Regions; ++r) {
#pragma unroll 1
        for (int c = 0; c < MPAD / 16; ++c) {
          float v[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) v[jj] = 0.0f;
#pragma unroll
          for (int e = 0; e < Cfg::kSets; ++e) {
            uint32_t u[16];
            tmem_ld16(tb + (e * kW4Regions + r) * MPAD + c * 16, u);
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) v[jj] += __uint_as_float(u[jj]);
          }
#pragma unroll
          for (int w = 0; w < 4; ++w)
            red[((r * (MPAD / 4)) + c * 4 + w) * 128 + tid] =
                make_float4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
        }
      }
    }
  }
  if (S > 1) cluster_sync_all();
  if (epi) {
    const int n = nb * kW4BN + 4 * tid;
    const int worker = static_cast<int>(rank) * 2 + g;
#pragma unroll 1
    for (int c = worker; c < kChunks; c += 2 * S) {
      float v[kW4Regions][8];
      if (S == 1) {
#pragma unroll
        for (int r = 0; r < kW4Regions; ++r) {
#pragma unroll
          for (int j = 0; j < 8; ++j) v[r][j] = 0.0f;
#pragma unroll
          for (int e = 0; e < Cfg::kSets; ++e) {
            uint32_t u[8];
            tmem_ld8(tb + (e * kW4Regions + r) * MPAD + c * 8, u);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j) v[r][j] += have ? __uint_as_float(u[j]) : 0.0f;
          }
        }
      } else if constexpr (!Cfg::kPush) {
#pragma unroll
        for (int r = 0; r < kW4Regions; ++r)
#pragma unroll
          for (int j = 0; j < 8; ++j) v[r][j] = 0.0f;
        for (int p = 0; p < S; ++p) {
#pragma unroll
          for (int r = 0; r < kW4Regions; ++r) {
#pragma unroll
            for (int w = 0; w < 2; ++w) {
              float4* src = &red[((r * (MPAD / 4)) + c * 2 + w) * 128 + tid];
              const float4 f = p == static_cast<int>(rank)
                                   ? *src
                                   : ld_dsmem_f4(mapa_shared(smem_u32(src),
                                                             static_cast<uint32_t>(p)));
              v[r][4 * w] += f.x;
              v[r][4 * w + 1] += f.y;
              v[r][4 * w + 2] += f.z;
              v[r][4 * w + 3] += f.w;
            }
          }
        }
      }
      const int64_t m0 = static_cast<int64_t>(mb) * MPAD + c * 8;
      switch (a.ep.act) {
        case kActRelu: epi_quad8<kActRelu>(v, m0, n, a.M, a.N, a.ep); break;
        case kActSilu: epi_quad8<kActSilu>(v, m0, n, a.M, a.N, a.ep); break;
        case kActGeluTanh: epi_quad8<kActGeluTanh>(v, m0, n, a.M, a.N, a.ep); break;
        default: epi_quad8<kActIdentity>(v, m0, n, a.M, a.N, a.ep); break;
      }
    }
  }
  // no rank leaves while another may still read its shared memory (every
  // remote load's value is used before its thread arrives: relaxed arrival)
  if (S > 1) cluster_sync_relaxed_arrive();
  }

  if (ctl.prof && threadIdx.x == 0) atomicAdd(&ctl.prof[31], static_cast<unsigned long long>(clock64() - t_start));
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

namespace {

template <int FMT, int MPAD>
cudaError_t run_w4(const GemmPlan& p, const CUtensorMap& tmA, const CUtensorMap& tmQ,
                   const CUtensorMap& tmS, const W4Args& args, int group, cudaStream_t stream) {
  using Cfg = W4Cfg<FMT, MPAD>;
  static std::atomic<uint64_t> mask{0};
  auto kernel = wq_gemm_kernel<FMT, MPAD>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(mask.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    mask.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.n_tiles, p.m_tiles);
  cfg.blockDim = dim3(kW4Threads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the previous kernel in the stream finishes (it waits
  // with griddepcontrol.wait before touching anything that kernel writes)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, tmA, tmQ, tmS, args, group);
}

}  // namespace

template <int FMT>
cudaError_t run_w4_fmt(const GemmPlan& plan, const CUtensorMap& tmA, const CUtensorMap& tmQ,
                       const CUtensorMap& tmS, const W4Args& args, int group,
                       cudaStream_t stream) {
  switch (plan.mpad) {
    case 16: return run_w4<FMT, 16>(plan, tmA, tmQ, tmS, args, group, stream);
    case 32: return run_w4<FMT, 32>(plan, tmA, tmQ, tmS, args, group, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_wq_gemm(int fmt, const GemmPlan& plan, const CUtensorMap& tmA,
                           const CUtensorMap& tmQ, const CUtensorMap& tmS, const EpiParams& ep,
                           int M, int N, int K, int group, const KernelCtl& ctl,
                           cudaStream_t stream) {
  W4Args args{M, N, K, plan.num_kb, plan.splits, ep, ctl};
  // the NVFP4 operand is the weight scaled by 2^-19 (deq_fp4_rowpair_scaled)
  if (fmt == kWqNvfp4) args.ep.alpha *= kNvfp4OperandScale;
  switch (fmt) {
    case kWqInt4: return run_w4_fmt<kWqInt4>(plan, tmA, tmQ, tmS, args, group, stream);
    case kWqFp8: return run_w4_fmt<kWqFp8>(plan, tmA, tmQ, tmS, args, group, stream);
    case kWqNvfp4: return run_w4_fmt<kWqNvfp4>(plan, tmA, tmQ, tmS, args, group, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gbf
