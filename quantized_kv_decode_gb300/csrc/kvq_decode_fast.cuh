// Tensor-core split-K decode attention over INT2/INT4/INT8 and NF4 caches
// (sm_103a).
//
// What it computes is the decode step of "Quantization & inference
// optimisation" ("Prefill, then decode": scores = K q / sqrt(d), softmax,
// weighted V over every cached row), with the keys and values read as
// group-wise codes and dequantized x_hat = (q - z) * s in registers
// ("What actually happens when you quantize a KV cache", sections 3-4 and 6).
//
// Structure (one CTA per (split, KV head, sequence); kWarps warps):
//  * Each warp streams its own 32-token tiles through a private cp.async
//    pipeline (16-byte chunks, zero-filled past the end of the sequence or
//    for unmapped pages) into shared memory whose code rows are XOR-swizzled
//    by 16-byte chunk, which makes every ldmatrix below free of bank
//    conflicts.
//  * Scores, mma.m16n8k16 (fp16 in, fp32 accumulate): A = q, one row per
//    (group, head) pair, holding that head's channels of that group only;
//    B = the codes of 8 tokens as exact fp16 subnormals c * 2^-24 (one AND
//    per code pair).  Row (g, h) of the accumulator is 2^-24 sum_{d in g}
//    q_h[d] c[d]; the epilogue forms s_g (sum - z_g sum_{d in g} q_h[d]) in
//    fp32, with the 2^24 in its scale, and adds the groups with warp
//    shuffles.  Token-rows shapes swap the operands (A = codes of 16
//    tokens, B = q).  Axis-aware caches keep K codes biased, 1024 + c, and
//    start the accumulator at minus the offset.
//  * Online softmax per 32-token tile (log2 domain), rescaling only when a
//    head's tile maximum exceeds its reference maximum by kSlack.
//  * Weighted V, mma.m16n8k16: A = V codes transposed (ldmatrix.trans puts
//    two tokens of one channel in each register) as subnormals (NF4: their
//    levels), B = p * s_g per token and group (fp16); the zero-points enter
//    through one extra mma per n-tile whose A rows hold z_g per token,
//    subtracted once at the end.
//  * The warps' (m, l, o) are merged in shared memory; the CTA writes the
//    final row (one split) or its partial for the merge kernel.
//  * Fused append (lens_before set): the CTA holding the new position
//    quantizes the new K/V in one warp, stores them, and merges the token as
//    one more partial; its tiles stop before that position.
#pragma once

#include "kvq_kivi.cuh"

namespace kvq {
namespace fast {

constexpr int kWarps = 4;
constexpr int kTT = 32;  // tokens per warp tile

template <int BITS, int D, int NG, int GP, bool KCH = false>
struct Cfg {
  static constexpr int ROWB = D * BITS / 8;       // code bytes per token row
  static constexpr int CHUNKS = ROWB / 16;        // 16-byte chunks per row
  static constexpr int RPL = 128 / ROWB;          // token rows per 128-byte line
  static constexpr int GSZ = D / NG;              // channels per group
  static constexpr int DPC = 128 / BITS;          // channels per 16-byte chunk
  static constexpr int KB = D / 16;               // k-blocks of the score mma
  static constexpr int MT = D / 16;               // m-tiles of the V mma
  static constexpr int HDRB = NG * 2;             // header bytes per token
  static constexpr int CODE_TILE = kTT * ROWB;
  static constexpr int HDR_TILE = kTT * HDRB;
  // K header bytes of a stage: per-token scale + zero rows, or (KCH, axis-
  // aware caches) the tile's block: one fp16 scale and zero per channel
  static constexpr int KHB = KCH ? 4 * D : 2 * HDR_TILE;
  static constexpr int STAGE = 2 * CODE_TILE + KHB + 2 * HDR_TILE;
  // per-warp scratch of the header pass, rows [group] of [token] entries
  // padded so that lanes reading different groups hit different banks:
  // fp32 K (scale * softmax scale in log2 units, zero) pairs, fp16 V scale,
  // fp16 V zero; then an fp32 [token] additive mask (0 or -inf)
  static constexpr int KROW = kTT + 8;            // float2 entries per K row
  static constexpr int VROW = kTT + 8;            // half entries per V row
  static constexpr int XHDR = NG * KROW * 8 + 2 * NG * VROW * 2 + kTT * 4;
  // Two CTAs per SM; as many stages (2..5) as then fit.  The header scratch
  // is double-buffered because tile i+1's scores are formed while tile i's
  // values are still being read.
  static constexpr int BUDGET = 110 * 1024 / kWarps;  // shared bytes per warp
  static constexpr int STAGES_FIT = (BUDGET - 2 * XHDR) / STAGE;
  static constexpr int STAGES = STAGES_FIT > 5 ? 5 : (STAGES_FIT < 2 ? 2 : STAGES_FIT);
  static constexpr int WARP_BYTES = STAGES * STAGE + 2 * XHDR;
  static constexpr int MIN_CTAS = 2;
  // Per-token caches with one query head per KV head, or INT4 token-rows
  // GQA shapes: a fifth warp does the fused step's append (quantize, store,
  // one-token partial) next to the four streaming warps instead of in front
  // of one of them's tiles.  (The other shapes need more registers than 160
  // threads leave for two CTAs per SM.)
  static constexpr bool AW = !KCH && (GP == 1 || (BITS == 4 && NG * GP <= 8));
  static constexpr int THREADS = kWarps * 32 + (AW ? 32 : 0);
  static constexpr int NTV = (NG * GP + 7) / 8;           // V-mma n-tiles: columns (group, head)
  static constexpr int NGL = (NG < 8 / GP) ? NG : 8 / GP;  // groups in accumulator rows 0..7
  static constexpr bool HI = NG * GP > 8;                   // rows 8..15 in use
  static_assert(BITS == 2 || BITS == 4 || BITS == 8, "bits");
  static_assert(BITS != 2 || !KCH, "INT2: per-token caches only");
  // INT2: a 16-byte chunk spans 64 channels; a chunk of more than one group
  // needs all its (group, head) columns in one V-mma n-tile
  static_assert(BITS != 2 || GSZ % DPC == 0 || NG * GP <= 8, "INT2 groups");
  static_assert(ROWB == 32 || ROWB == 64 || ROWB == 128, "code row size");
  static_assert(BITS == 2 || GSZ % DPC == 0, "a 16-byte chunk must lie inside one group");
  static_assert(NG * GP <= 16, "groups x padded heads must fit 16 rows");
  static_assert(HDRB == 4 || HDRB == 8 || HDRB == 16, "header row size");
  static_assert(2 * GP * (D + 2) * 4 <= WARP_BYTES, "the CTA merge reuses the pipeline region");
  static_assert(!KCH || NG * KROW * 8 >= 4 * D, "KCH: block header scratch");

  // Shared-memory byte offset of 16-byte chunk c of token row t: chunk slots
  // are XOR-swizzled by the row's position so that the 8 rows an ldmatrix
  // reads at one chunk index fall in 8 different 16-byte bank groups.
  __device__ static __forceinline__ uint32_t at(int t, int c) {
    return (uint32_t)(t * ROWB + ((c ^ ((t / RPL) & (CHUNKS - 1))) << 4));
  }
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_small(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;\n" ::"r"(dst), "l"(src), "n"(N),
               "r"(valid ? N : 0)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}

__device__ __forceinline__ void ldsm_x2(uint32_t a, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r0), "=r"(r1)
               : "r"(a));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// fp16 bit patterns: 1024 and 1/16 in both halves
constexpr uint32_t kH1024 = 0x64006400u;
constexpr uint32_t kH1_16 = 0x2C002C00u;

// (a & b) | c in one LOP3
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Eight 4-bit codes of one 32-bit word (code k in bits 4k..4k+3) to four
// biased fp16 pairs: (0x6400 | c) is the fp16 value 1024 + c, (0x6400 | 16c)
// is 1024 + 16c; o[0] = (1024+c0, 1024+c4), o[1] = (1024+16c1, 1024+16c5),
// o[2] = (1024+c2, 1024+c6), o[3] = (1024+16c3, 1024+16c7).  The axis-aware
// caches' K side uses them: the accumulator's starting value removes the
// offset, and q/16 in the matching slots undoes the x16.
__device__ __forceinline__ void nib8_to_h2_biased(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t w2 = w >> 8;
  o[0] = and_or(w, 0x000F000Fu, kH1024);
  o[1] = and_or(w, 0x00F000F0u, kH1024);
  o[2] = and_or(w2, 0x000F000Fu, kH1024);
  o[3] = and_or(w2, 0x00F000F0u, kH1024);
}

// The same codes as exact fp16 subnormals: with no exponent bits the half
// (c) is c * 2^-24 and (16c) is 16c * 2^-24, so the contractions carry no
// offset; the 2^24 goes into a scale on the other side of each contraction.
// mma.sync takes fp16 subnormal operands without flushing them to zero; every
// parity test of the tensor-core path depends on that.
__device__ __forceinline__ void nib8_to_h2_sub(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t w2 = w >> 8;
  o[0] = w & 0x000F000Fu;
  o[1] = w & 0x00F000F0u;
  o[2] = w2 & 0x000F000Fu;
  o[3] = w2 & 0x00F000F0u;
}

// prmt.b32 in its default mode: a selector nibble with bit 3 set gives its
// output byte the sign (bit 7) of the selected byte, replicated.
__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// NF4 codes of one 32-bit word to their fp16 levels, in the pairing of
// nib8_to_h2_biased: o[0] = (lv(c0), lv(c4)), o[1] = (lv(c1), lv(c5)), ...
// The 16 levels are antisymmetric, lv(15 - c) = -lv(c), so a code picks one
// of 8 magnitudes (c - 8 for c >= 8, 7 - c below) and a sign.  lut holds
// the magnitudes' fp16 bytes: lut[0] / lut[1] the low bytes of magnitudes
// 0-3 / 4-7, lut[2] / lut[3] the high bytes; byte permutes do the lookup,
// and sign-replicating permutes of the codes' bit 3 set the sign bits.
__device__ __forceinline__ void nib8_to_h2_nf4(uint32_t w, uint32_t (&o)[4],
                                               const uint32_t (&lut)[4]) {
  const uint32_t S = ~w & 0x88888888u;                         // per code: bit 3 set iff lv < 0
  const uint32_t idx = (w ^ (S - (S >> 3))) & 0x77777777u;      // magnitude index
  const uint32_t S4 = S << 4;  // the flags of even codes at their byte's bit 7
  const uint32_t s01 = prmt_b32(idx, 0u, 0x0020u);  // selectors (c0, c1, c4, c5)
  const uint32_t s23 = prmt_b32(idx, 0u, 0x0031u);  // selectors (c2, c3, c6, c7)
  const uint32_t pl = prmt_b32(lut[0], lut[1], s01);
  const uint32_t ql = prmt_b32(lut[0], lut[1], s23);
  const uint32_t ph = prmt_b32(lut[2], lut[3], s01) | (prmt_b32(S4, S, 0xEAC8u) & 0x80808080u);
  const uint32_t qh = prmt_b32(lut[2], lut[3], s23) | (prmt_b32(S4, S, 0xFBD9u) & 0x80808080u);
  o[0] = prmt_b32(pl, ph, 0x6240u);
  o[1] = prmt_b32(pl, ph, 0x7351u);
  o[2] = prmt_b32(ql, qh, 0x6240u);
  o[3] = prmt_b32(ql, qh, 0x7351u);
}

// Sixteen 2-bit codes (byte m = codes 4m .. 4m+3, code 4m + f in bits 2f of
// byte m) to fp16 subnormal pairs 4^f c * 2^-24, f = k & 3, one AND each:
// o[k] = (code at byte k>>2, field f; the same field of byte 2 + (k>>2)).
// The factor 4^f is undone on the other operand (score side) or at the end
// (value side).
__device__ __forceinline__ void crumb16_to_h2_sub(uint32_t w, uint32_t (&o)[8]) {
  const uint32_t w2 = w >> 8;
#pragma unroll
  for (int f = 0; f < 4; ++f) {
    o[f] = w & (0x00030003u << (2 * f));
    o[4 + f] = w2 & (0x00030003u << (2 * f));
  }
}

// The 4-bit conversion of a kernel instance: NF4 levels, subnormal codes or
// (axis-aware K) biased codes.
template <bool NF, bool SUB>
__device__ __forceinline__ void nib8_to_h2(uint32_t w, uint32_t (&o)[4], const uint32_t (&lut)[4]) {
  if constexpr (NF) nib8_to_h2_nf4(w, o, lut);
  else if constexpr (SUB) nib8_to_h2_sub(w, o);
  else nib8_to_h2_biased(w, o);
}

// Four 8-bit codes (byte k = code k) to fp16 pairs 1024 + c (score side),
// or (SUB) the subnormals c * 2^-24.
template <uint32_t SEL, bool SUB = false>
__device__ __forceinline__ uint32_t byte2_to_h2_biased(uint32_t w) {
  return __byte_perm(w, SUB ? 0u : 0x64646464u, SEL);
}

// Four 8-bit codes (byte k = code k) to fp16 subnormal pairs c * 2^-24 per
// the selectors: 0x4240 -> (c0, c2), 0x4341 -> (c1, c3) (value side).
template <uint32_t SEL>
__device__ __forceinline__ uint32_t byte2_to_h2_sub(uint32_t w) {
  return __byte_perm(w, 0u, SEL);
}

// 2^x by the SFU (flush-to-zero; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Pull [p, p + bytes) into L2 (p and bytes multiples of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  return h2_as_u32(__floats2half2_rn(lo, hi));
}

__device__ __forceinline__ uint32_t pack_halves(__half lo, __half hi) {
  return h2_as_u32(__halves2half2(lo, hi));
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

// Dynamic shared memory of an instance: q, the warps' pipelines (reused by
// the CTA merge), the tile masks and the appended token's partial; NF4
// instances then hold their score-side level table (kNfLutBytes, 16-byte
// aligned).
template <int BITS, int D, int NG, int GP, bool KCH>
__host__ __device__ constexpr size_t fast_smem_bytes() {
  using C = Cfg<BITS, D, NG, GP, KCH>;
  const size_t pipe = (size_t)kWarps * C::WARP_BYTES;
  const size_t masks = ((kWarps * C::STAGES * 4 + 15) / 16) * 16;
  const size_t newtok = (D + GP) * sizeof(float);
  const size_t merge = (size_t)kWarps * GP * (D + 2) * sizeof(float) * (KCH ? 2 : 1);
  return ((GP * D * 2 + 127) / 128) * 128 + (pipe > merge ? pipe : merge) + masks + newtok;
}

// NF4 score side: a table of the fp16 level pairs of every code byte (low
// nibble = even channel), one word per byte value, in kNfLutCopies copies
// interleaved word by word so that lanes of different copies never share a
// bank for the same byte value.
constexpr int kNfLutCopies = 8;
constexpr size_t kNfLutBytes = 256 * kNfLutCopies * 4;
template <int BITS, int D, int NG, int GP, bool KCH>
__host__ __device__ constexpr size_t nf_lut_offset() {
  return (fast_smem_bytes<BITS, D, NG, GP, KCH>() + 15) / 16 * 16;
}

// NF4 codes of one 32-bit word to their fp16 levels through that table,
// byte by byte: o[k] = (level(low nibble), level(high nibble)) of byte k.
// lut_lane: shared-memory address of this lane's copy.
__device__ __forceinline__ void nib8_to_h2_nf4_table(uint32_t w, uint32_t (&o)[4],
                                                     uint32_t lut_lane) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t byte;  // byte k of w, zero-extended
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(byte) : "r"(w), "r"(0x4440u + k));
    // (the table is written before the barrier that precedes every tile,
    // and w comes from a tile, so the load cannot move ahead of it)
    asm("ld.shared.u32 %0, [%1];" : "=r"(o[k]) : "r"(lut_lane + byte * (uint32_t)(kNfLutCopies * 4)));
  }
}

// Threshold (log2 units) by which a head's tile maximum may exceed the
// reference maximum before the accumulators are rescaled; probabilities are
// bounded by 2^kSlack.
constexpr float kSlack = 4.f;

template <int BITS, int D, int NG, int GP, bool SYM, bool KCH, bool NF = false, bool PG = false>
__global__ void __launch_bounds__(Cfg<BITS, D, NG, GP, KCH>::THREADS, Cfg<BITS, D, NG, GP, KCH>::MIN_CTAS)
    decode_fast_kernel(const DecodeParams p) {
  // SYM: symmetric caches, no zero arrays; every zero-point is 2^(BITS-1).
  // NF: NF4 codes (with SYM: scale only), which stand for normal-quantile
  // levels; no offset to remove and no zero-point.
  static_assert(!NF || (BITS == 4 && SYM && !KCH), "NF4: 4-bit, scale-only, per-token");
  // PG: a paged axis-aware cache (kch_row / kch_hdr map its rows; the dense
  // instances keep their own addressing)
  static_assert(!PG || KCH, "PG: axis-aware caches");
  constexpr unsigned short kSymZero =
      NF ? 0u : (BITS == 2 ? 0x4000u : (BITS == 4 ? 0x4800u : 0x5800u));  // fp16 0, 2, 8, 128
  // Integer codes enter the tensor cores as fp16 subnormals (code * 2^-24,
  // see nib8_to_h2_sub): no offsets to cancel.  kSubK / kSubV restore the
  // scale: the K scales in the header scratch and the q sums of the
  // zero-point term carry kSubK (axis-aware caches: the score epilogue),
  // the final rows kSubV.  Axis-aware caches in the (group, head)-rows
  // layout keep biased K codes, whose offset their accumulators start at.
  constexpr bool SUBK = !NF && (!KCH || GP == 1);
  constexpr float kSubK = SUBK ? 16777216.f : 1.f;  // 2^24
  constexpr float kSubV = NF ? 1.f : 16777216.f;
  const float kscale = p.scale_log2 * kSubK;  // K scale factor of the header scratch
  // NF4, value side: the 8 level magnitudes as fp16 bytes (see nib8_to_h2_nf4)
  uint32_t lut[4] = {0u, 0u, 0u, 0u};
  if constexpr (NF) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t hb = __half_as_ushort(__float2half_rn(p.nf4_level[8 + k]));
      lut[k >> 2] |= (hb & 0xFFu) << (8 * (k & 3));
      lut[2 + (k >> 2)] |= (hb >> 8) << (8 * (k & 3));
    }
  }
  using C = Cfg<BITS, D, NG, GP, KCH>;
  extern __shared__ __align__(128) uint8_t smem[];
  // NF4: the score side's level table (see nib8_to_h2_nf4_table), built
  // from the kernel's own parameters before the wait; the barrier after q is
  // staged publishes it
  uint32_t nf_lut_lane = 0u;
  if constexpr (NF) {
    uint32_t* t = reinterpret_cast<uint32_t*>(smem + nf_lut_offset<BITS, D, NG, GP, KCH>());
    for (int i = threadIdx.x; i < 256 * kNfLutCopies; i += blockDim.x) {
      const int v = i / kNfLutCopies;
      t[i] = pack_halves(__float2half_rn(p.nf4_level[v & 15]), __float2half_rn(p.nf4_level[v >> 4]));
    }
    nf_lut_lane = smem_u32(t + (threadIdx.x & (kNfLutCopies - 1)));
  }
  // Token-rows layout, whenever the (group, head) pairs fill at most 8 rows
  // of the (group, head)-rows layout: the score mma takes the codes as A
  // (rows = 16 tokens) and q as B (columns = (group, head) pairs), half the
  // mmas.  The scores are then moved into the lanes the softmax and the V
  // side expect.  Axis-aware caches use it for one query head per KV head.
  // With 16 (group, head) pairs (TQ2: GP = 2 or 4) the columns span two
  // n-tiles, each k-block's group lying in one of them, so a k-block still
  // takes one mma per 16 tokens: n-tile 1 holds the pairs of rows 8..15.
  constexpr bool TQ2 = !KCH && BITS != 2 && (GP == 2 || GP == 4) && NG * GP == 16;
  constexpr bool TQ = GP == 1 || (!KCH && GP <= 4 && NG * GP <= 8) || TQ2;
  // the q n-tile of k-block kb's group (TQ2), else 0
  auto qtile = [](int kb) { return TQ2 ? ((kb * 16) / C::GSZ) / (8 / GP) : 0; };
  const CacheGeom& geo = p.geom;
  const int split = blockIdx.x, kvh = blockIdx.y;
  const int G = p.G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rho = lane >> 2, j = lane & 3;

  // Launched with programmatic stream serialization: the next kernel of the
  // stream may start launching now.  Until the previous kernel has completed
  // (pdl_wait) nothing here reads or writes caller memory; it only warms L2
  // with this warp's first tiles (dense caches, as if the sequence filled the
  // cache), the CTA's q rows and the new token's K/V rows.  Those bytes are
  // read again after the wait, so a previous kernel that wrote them is still
  // seen.
  pdl_launch_dependents();
  if constexpr (!KCH) {
    if (!p.longest_first && geo.layout == KVQ_DENSE && warp < kWarps && lane < C::STAGES * 6) {
      const int b = blockIdx.z;
      const int it = lane / 6, region = lane % 6;
      const int t0g = split * p.chunk;
      const int t1g = min(geo.slots, t0g + p.chunk);
      const int start = t0g + (warp + it * kWarps) * kTT;
      if (start < t1g && !(SYM && (region == 3 || region == 5))) {
        const int n = min(kTT, t1g - start);
        const long long row0 = ((long long)b * geo.Hkv + kvh) * geo.slots + start;
        const int per = region < 2 ? C::ROWB : C::HDRB;
        const void* base = region == 0 ? (const void*)p.codes[0] : region == 1 ? (const void*)p.codes[1]
                         : region == 2 ? (const void*)p.scale[0] : region == 3 ? (const void*)p.zero[0]
                         : region == 4 ? (const void*)p.scale[1] : (const void*)p.zero[1];
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(base) + (uintptr_t)(row0 * per);
        const uintptr_t a1 = a0 + (uintptr_t)n * per;
        const uintptr_t lo = a0 & ~(uintptr_t)15, hi = a1 & ~(uintptr_t)15;  // stay inside the array
        // (region r is kvq_array r: K / V codes, K scale / zero, V scale / zero)
        if (hi > lo && KVQ_IN(geo, region, reinterpret_cast<const void*>(lo), hi - lo))
          prefetch_l2(reinterpret_cast<const void*>(lo), (uint32_t)(hi - lo));
      }
    }
  }
  // the CTA's q rows, for the fused step the new token's K and V rows, and
  // for axis-aware caches the unit's fp16 rows (sinks and residual window)
  if (!p.longest_first && warp == 1 && lane < 5) {
    const int b = blockIdx.z;
    const void* src = nullptr;
    uint32_t bytes = 0;
    const int arr = lane == 0 ? KVQ_ARRAY_Q : lane < 3 ? KVQ_ARRAY_K_NEW + (lane - 1)
                                                       : KVQ_ARRAY_K_WINDOW + (lane - 3);
    if (lane == 0) {
      src = p.q + ((long long)b * p.Hq + (long long)kvh * G) * D;
      bytes = (uint32_t)(G * D * 2);
    } else if (lane < 3) {
      if (p.lens_before != nullptr) {
        src = p.new_kv[lane - 1] + ((long long)b * geo.Hkv + kvh) * D;
        bytes = (uint32_t)(D * 2);
      }
    } else if (KCH) {
      src = p.window[lane - 3] + ((long long)b * geo.Hkv + kvh) * (geo.sink + geo.g) * D;
      bytes = (uint32_t)((geo.sink + geo.g) * D * 2);
    }
    if (src != nullptr && (reinterpret_cast<uintptr_t>(src) & 15) == 0 && KVQ_IN(geo, arr, src, bytes))
      prefetch_l2(src, bytes);
  }
  // Longest-first grids learn their sequence only after the wait, so their
  // CTAs cannot warm their own rows: the first three CTAs warm L2 with the
  // whole q array and the new K and V rows instead, in 32 slices each
  // (GQA mix 66.48 -> 66.06 us per fused call)
  if (p.longest_first && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z < 3 && warp == 1) {
    const int z = blockIdx.z;
    const void* base = z == 0 ? (const void*)p.q
                     : (p.lens_before != nullptr ? (const void*)p.new_kv[z - 1] : nullptr);
    const unsigned long long total = (unsigned long long)p.batch * (z == 0 ? p.Hq : geo.Hkv) * D * 2;
    const unsigned long long slice = ((total + 31) / 32 + 15) / 16 * 16;
    const unsigned long long lo = slice * lane;
    if (base != nullptr && (reinterpret_cast<uintptr_t>(base) & 15) == 0 && lo < total) {
      const unsigned long long n = (total - lo < slice ? total - lo : slice) / 16 * 16;
      const uint8_t* from = reinterpret_cast<const uint8_t*>(base) + lo;
      if (n > 0 && KVQ_IN(geo, z == 0 ? KVQ_ARRAY_Q : KVQ_ARRAY_K_NEW + (z - 1), from, n))
        prefetch_l2(from, (uint32_t)n);
    }
  }
  pdl_wait();

  const int b = p.longest_first ? longest_first_seq(p, blockIdx.z, reinterpret_cast<int*>(smem))
                                : (int)blockIdx.z;
  int L = seq_len_of(p, b);
  if (L < 0 || L > p.len_limit) {
    if (threadIdx.x == 0 && split == 0 && kvh == 0 && p.status) atomicOr(p.status, KVQ_FLAG_SEQ_LEN);
    L = 0;
  }
  const int t0 = split * p.chunk;
  const int t1 = min(L, t0 + p.chunk);
  if (p.splits > 1 && t0 >= L) {
    // no tokens in this split: the merge skips it by its m = -inf
    if (p.merge_all && threadIdx.x < G) {
      float* mlo = p.ws_ml + (((long long)b * p.Hq + (long long)kvh * G + threadIdx.x) * p.splits + split) * 2;
      if (KVQ_IN(geo, KVQ_ARRAY_WORKSPACE, mlo, 8)) {
        mlo[0] = -INFINITY;
        mlo[1] = 0.f;
      }
    }
    return;
  }
  // Longest-first grids learn their sequence only here: warm the new K/V
  // rows a fused step's append reads while q is staged.
  if (!KCH && p.longest_first && p.lens_before != nullptr && L > 0 && L - 1 >= t0 && L - 1 < t1 &&
      threadIdx.x < 2) {
    const __half* src = p.new_kv[threadIdx.x] + ((long long)b * geo.Hkv + kvh) * D;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0 &&
        KVQ_IN(geo, KVQ_ARRAY_K_NEW + (int)threadIdx.x, src, D * 2))
      prefetch_l2(src, (uint32_t)(D * 2));
  }

  // shared memory: [q fp16 GP x D][per warp: stages, header scratch][tile
  // masks][the appended token's partial: v_hat fp32 [D], scores fp32 [GP]]
  __half* q_s = reinterpret_cast<__half*>(smem);
  uint8_t* pipe = smem + ((GP * D * 2 + 127) / 128) * 128;
  uint32_t* mask_s = reinterpret_cast<uint32_t*>(pipe + kWarps * C::WARP_BYTES);
  float* tok_v = reinterpret_cast<float*>(pipe + kWarps * C::WARP_BYTES +
                                         ((kWarps * C::STAGES * 4 + 15) / 16) * 16);
  float* tok_s = tok_v + D;
  uint8_t* wpipe = pipe + warp * C::WARP_BYTES;
  // header scratch buffer `buf` (0/1): K (s*scale, z) [NG][KROW], V scale
  // [NG][VROW], V zero [NG][VROW], token mask [kTT]
  uint8_t* xbase = wpipe + C::STAGES * C::STAGE;
  auto ksz_of = [&](int buf) { return reinterpret_cast<float2*>(xbase + buf * C::XHDR); };
  auto vsx_of = [&](int buf) { return reinterpret_cast<__half*>(ksz_of(buf) + NG * C::KROW); };
  auto vzx_of = [&](int buf) { return vsx_of(buf) + NG * C::VROW; };
  auto madd_of = [&](int buf) { return reinterpret_cast<float*>(vzx_of(buf) + NG * C::VROW); };

  const __half* qg = p.q + ((long long)b * p.Hq + (long long)kvh * G) * D;
  for (int i = threadIdx.x; i < GP * D; i += blockDim.x)
    q_s[i] = (i < G * D && KVQ_IN(geo, KVQ_ARRAY_Q, qg + i, 2)) ? qg[i] : __float2half_rn(0.f);
  // Fused step on an axis-aware cache, one split: this CTA appends its
  // unit's new token (position L - 1) with the append kernel's code, so that
  // it reads the cache as the two-call step leaves it.  A token that
  // completes its block has the block quantized here, before any tile is
  // copied (the fence makes the codes visible to the L2-only copies); a token
  // bound for an fp16 slot (a sink or the residual ring) is read from the
  // input by the window pass and stored to its slot at the end.
  int kch_slot = -1;  // the new token's window slot, or -1
  if constexpr (KCH && BITS != 2) {
    if (p.kch_append && L > 0) {
      const int p0 = L - 1;
      kch_slot = window_slot(geo, L, p0);
      if (kch_slot < 0) {
        KiviIO io;
        io.geom = &geo;
        for (int w = 0; w < 2; ++w) {
          io.codes[w] = const_cast<uint8_t*>(p.codes[w]);
          io.scale[w] = const_cast<__half*>(p.scale[w]);
          io.zero[w] = const_cast<__half*>(p.zero[w]);
          io.src[w] = p.new_kv[w];
          io.window[w] = const_cast<__half*>(p.window[w]);
        }
        io.status = p.status;
        io.num_new = 1;
        const int j = (p0 - geo.sink) / geo.g;
        kivi_quantize_block<BITS>(io, b, kvh, j, (long long)geo.sink + (long long)j * geo.g, p0);
        __threadfence();
      }
    }
  }

  __syncthreads();

  // Fused append: in the CTA whose range holds the new position, the tiles
  // stop short of it.  One warp quantizes the new K and V vectors (the
  // quantize8 the append kernel runs), stores them to the cache, and turns
  // the dequantized token into a one-token partial (score per head, weight
  // 1, value v_hat) that the CTA merge adds to the warps' partials.  No read
  // of this launch touches the new row, so the store needs no ordering.
  const int pos_new = L - 1;
  const bool owner_cta = !KCH && p.lens_before != nullptr && L > 0 && pos_new >= t0 && pos_new < t1;
  const int t_end = owner_cta ? t1 - 1 : t1;  // tiles cover [t0, t_end)

  // ---- score-mma A fragments: row r <-> (group r / GP, head r % GP); for
  // axis-aware caches (KCH) every row r holds head r % GP over all channels,
  // and the block's per-channel scales are multiplied in per tile ----
  const int g_lo = rho / GP, h_row = rho % GP;
  const int g_hi = g_lo + 8 / GP;
  const bool row_ok = h_row < G;
  // channel of the score-mma k-slots 2jj, 2jj+1, 2jj+8, 2jj+9 of k-block kb
  // (the order in which the code conversions deliver channels)
  auto slot_channels = [](int kb, int jj, int (&dk)[4]) {
    if constexpr (BITS == 2) {
      // k-block kb = 4 c + i of chunk c takes conversion outputs 2i, 2i+1
      const int i = kb & 3;
      const int x = 64 * (kb >> 2) + 16 * jj + 4 * (i >> 1) + 2 * (i & 1);
      dk[0] = x; dk[1] = x + 8; dk[2] = x + 1; dk[3] = x + 9;
    } else if constexpr (BITS == 4 && NF) {
      // the table conversion: byte k of the lane's word holds channels 2k, 2k + 1
      const int base = 32 * (kb >> 1) + 8 * jj + 4 * (kb & 1);
      dk[0] = base; dk[1] = base + 1; dk[2] = base + 2; dk[3] = base + 3;
    } else if constexpr (BITS == 4) {
      const int base = 32 * (kb >> 1) + 8 * jj + 2 * (kb & 1);
      dk[0] = base; dk[1] = base + 4; dk[2] = base + 1; dk[3] = base + 5;
    } else {
      const int base = 16 * kb + 4 * jj;
      dk[0] = base; dk[1] = base + 1; dk[2] = base + 2; dk[3] = base + 3;
    }
  };
  uint32_t qa[C::KB][4];
#pragma unroll
  for (int kb = 0; kb < C::KB; ++kb) {
    int dk[4];  // channel of k-slots 2j, 2j+1, 2j+8, 2j+9
    slot_channels(kb, j, dk);
    const int grp = dk[0] / C::GSZ;  // the four lie in one group
    const __half* qh = q_s + h_row * D;
    const bool lo = row_ok && (KCH || g_lo == grp);
    const bool hi = row_ok && (KCH || (C::HI && g_hi == grp));
    const uint32_t v01 = pack_halves(qh[dk[0]], qh[dk[1]]);
    uint32_t v23 = pack_halves(qh[dk[2]], qh[dk[3]]);
    uint32_t v01s = v01;
    if constexpr (BITS == 4 && !NF)  // slots 2j+8, 2j+9 meet the odd nibbles, held as 16c
      v23 = h2_as_u32(__hmul2(u32_as_h2(v23), u32_as_h2(kH1_16)));
    if constexpr (BITS == 2) {  // slots meet codes held as 4^f c: f = 2 (kb & 1), + 1 for 2j+8, 2j+9
      v01s = h2_as_u32(__hmul2(u32_as_h2(v01), u32_as_h2((kb & 1) ? kH1_16 : 0x3C003C00u)));
      v23 = h2_as_u32(__hmul2(u32_as_h2(v23), u32_as_h2((kb & 1) ? 0x24002400u : 0x34003400u)));
    }
    qa[kb][0] = lo ? v01s : 0u;
    qa[kb][1] = hi ? v01s : 0u;
    qa[kb][2] = lo ? v23 : 0u;
    qa[kb][3] = hi ? v23 : 0u;
  }
  // Per row (g, h): the sum of q_h over group g (the zero-point term), by an
  // mma against constant codes.
  float qs_lo = 0.f, qs_hi = 0.f, qs_lo1 = 0.f, qs_hi1 = 0.f;  // *1: TQ2's n-tile 1
  if constexpr (TQ) {
    // B = q: per column (group) 2j and 2j+1 of this lane, the sum of q over
    // the group
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    constexpr uint32_t kOnes = 0x3C003C00u;
    constexpr uint32_t kHi = (BITS == 4 && !NF) ? 0x4C004C00u : 0x3C003C00u;  // x16 undoes q/16 in odd slots
#pragma unroll
    for (int kb = 0; kb < C::KB; ++kb) {
      // INT2: 4^f undoes the slots' 4^-f (1, 4 or 16, 64)
      const uint32_t ulo = BITS == 2 ? ((kb & 1) ? 0x4C004C00u : kOnes) : kOnes;
      const uint32_t uhi = BITS == 2 ? ((kb & 1) ? 0x54005400u : 0x44004400u) : kHi;
      mma16816(acc, ulo, ulo, uhi, uhi, qa[kb][0], qa[kb][2]);
      if constexpr (TQ2) mma16816(acc1, ulo, ulo, uhi, uhi, qa[kb][1], qa[kb][3]);
    }
    qs_lo = acc[0];   // column 2j
    qs_hi = acc[1];   // column 2j + 1
    qs_lo1 = acc1[0];
    qs_hi1 = acc1[1];
  } else if constexpr (!KCH) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    constexpr uint32_t kOnes = 0x3C003C00u;   // fp16 (1, 1)
    constexpr uint32_t kSixteen = 0x4C004C00u;  // fp16 (16, 16)
#pragma unroll
    for (int kb = 0; kb < C::KB; ++kb) {
      const uint32_t ulo = BITS == 2 ? ((kb & 1) ? kSixteen : kOnes) : kOnes;
      const uint32_t uhi = BITS == 2 ? ((kb & 1) ? 0x54005400u : 0x44004400u)
                                     : ((BITS == 4 && !NF) ? kSixteen : kOnes);
      mma16816(acc, qa[kb][0], qa[kb][1], qa[kb][2], qa[kb][3], ulo, uhi);
    }
    qs_lo = acc[0];
    qs_hi = acc[2];
  }
  // subnormal codes: the score accumulators carry 2^-24 sum q c, so the
  // zero-point term's q sums do too (the header's K scales carry 2^24)
  qs_lo *= 1.f / kSubK;
  qs_hi *= 1.f / kSubK;
  qs_lo1 *= 1.f / kSubK;
  qs_hi1 *= 1.f / kSubK;
  const int g_lo_c = min(g_lo, NG - 1), g_hi_c = min(g_hi, NG - 1);
  // After the group sum, lane rho holds the scores of head rho % GP; lanes of
  // a head beyond G read a row of -inf as their token mask.
  const int h_lane = rho % GP;
  const float hmask = (h_lane < G) ? 0.f : -INFINITY;
  // V-mma B columns of this lane, per n-tile t: (group (8t + rho) / GP, head h_lane)
  int gcol[C::NTV];
#pragma unroll
  for (int t = 0; t < C::NTV; ++t) gcol[t] = (8 * t + rho) / GP;

  // ---- running state ----
  float o[C::MT][4];
#pragma unroll
  for (int m = 0; m < C::MT; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
  float cz[C::NTV][4];  // zero-point terms: rows = groups r, columns = (group, head)
#pragma unroll
  for (int t = 0; t < C::NTV; ++t) cz[t][0] = cz[t][1] = cz[t][2] = cz[t][3] = 0.f;
  bool bt_bad = false;  // an unmapped page was met (flagged once at the end)
  float m_ref = -INFINITY, l_run = 0.f;

  // ---- this warp's tiles ----
  // KCH: sinks [0, kS) and the residual window [kr0, L) are fp16 and handled
  // after the loop; the tiles are the quantized blocks' 32-token tiles
  // (anchored at kS) whose first token lies in [t0, t1).
  int kS = 0, kr0 = 0, qbase = t0, ntiles;
  if constexpr (KCH) {
    kS = min(geo.sink, L);
    kr0 = kS + ((L - kS) / geo.g) * geo.g;
    const int m_lo = t0 <= kS ? 0 : (t0 - kS + kTT - 1) / kTT;
    const int m_hi = min((kr0 - kS) / kTT, t1 <= kS ? 0 : (t1 - kS + kTT - 1) / kTT);
    ntiles = max(0, m_hi - m_lo);
    qbase = kS + kTT * m_lo;
  } else {
    ntiles = (t_end > t0) ? (t_end - t0 + kTT - 1) / kTT : 0;
  }
  // the appending warp: one with the fewest tiles
  // (the append warp when the CTA has one)
  const int owner_warp = C::AW ? kWarps : ntiles % kWarps;
  const bool owner = owner_cta && warp == owner_warp;  // warp-uniform
  // Tiles go round-robin over the streaming warps.  In a fused step's owner
  // CTA without an append warp, the owner warp appends before it streams;
  // the last kSpill tiles (or all, in a short range) then go round-robin
  // over the other three warps only, so that the owner has about kSpill / 4
  // fewer tiles to make up for the append's time, about four tiles' worth
  // (a paged small-model CTA finished about 3 us later than with a
  // decode-only call).
  constexpr int kSpill = 12;
  const int spill = (owner_cta && !C::AW) ? min(kSpill, ntiles) : 0;
  const int nrr = ntiles - spill;  // tiles [0, nrr) round-robin over all streaming warps
  int nmine = (warp < kWarps && nrr > warp) ? (nrr - warp + kWarps - 1) / kWarps : 0;
  const int srank = warp - (warp > owner_warp ? 1 : 0);  // rank among the non-owner warps
  if (spill && warp < kWarps && warp != owner_warp)
    nmine += (spill - srank + kWarps - 2) / (kWarps - 1);
  // the CTA tile this warp takes as its it-th
  auto tile_of = [&](int it) {
    const int r = nrr > warp ? (nrr - warp + kWarps - 1) / kWarps : 0;
    return it < r ? warp + it * kWarps : nrr + srank + (it - r) * (kWarps - 1);
  };
  const uint8_t* kc_g = p.codes[0];
  const uint8_t* vc_g = p.codes[1];
  const uint8_t* ks_g = reinterpret_cast<const uint8_t*>(p.scale[0]);
  const uint8_t* kz_g = reinterpret_cast<const uint8_t*>(p.zero[0]);
  const uint8_t* vs_g = reinterpret_cast<const uint8_t*>(p.scale[1]);
  const uint8_t* vz_g = reinterpret_cast<const uint8_t*>(p.zero[1]);
  const bool dense = geo.layout == KVQ_DENSE;
  const long long slab_row = ((long long)b * geo.Hkv + kvh) * geo.slots;  // dense only
  const long long bt_row = (long long)b * geo.max_blocks;                 // paged only
  const bool pg_pow2 = (geo.slots & (geo.slots - 1)) == 0;
  const int pg_shift = __ffs(geo.slots) - 1;
  const uint32_t wpipe_s = smem_u32(wpipe);

  // issues tile `it` into its stage; returns true when a page was unmapped
  auto issue = [&](int it) -> bool {
    const int stage = it % C::STAGES;
    bool unmapped = false;
    if (it < nmine) {
      const int start = qbase + tile_of(it) * kTT;
      const int n = KCH ? kTT : min(kTT, t_end - start);
      long long row = -1;  // this lane's token
      const uint32_t kc_s = wpipe_s + stage * C::STAGE, vc_s = kc_s + C::CODE_TILE;
      const uint32_t hd_s = vc_s + C::CODE_TILE;
      if (dense) {
        if (lane < n) row = slab_row + start + lane;
        const long long base = (slab_row + start) * C::ROWB;
#pragma unroll
        for (int k = 0; k < C::CHUNKS; ++k) {
          const int c = lane + 32 * k;
          const int tok = c / C::CHUNKS, part = c % C::CHUNKS;
          const bool ok = tok < n;
          const long long off = ok ? base + tok * C::ROWB + part * 16 : 0;
          const uint32_t dst = C::at(tok, part);
          cp_async16(kc_s + dst, kc_g + off, ok && KVQ_IN(geo, KVQ_ARRAY_K_CODES, kc_g + off, 16));
          cp_async16(vc_s + dst, vc_g + off, ok && KVQ_IN(geo, KVQ_ARRAY_V_CODES, vc_g + off, 16));
        }
      } else if (!PG && p.rows32) {
        // rows and byte offsets in 32 bits; pages of a power-of-two size by a
        // shift
        int row32 = -1;
        if (lane < n) {
          const int pos = start + lane;
          const int blk = pg_pow2 ? pos >> pg_shift : pos / geo.slots;
          const int32_t* bte = geo.block_table + bt_row + blk;
          const int pg = KVQ_IN(geo, KVQ_ARRAY_BLOCK_TABLE, bte, 4) ? __ldg(bte) : -1;
          if (pg >= 0 && pg < geo.num_pages) row32 = (pg * geo.Hkv + kvh) * geo.slots + (pos - blk * geo.slots);
          unmapped = row32 < 0;
        }
        row = row32;
#pragma unroll
        for (int k = 0; k < C::CHUNKS; ++k) {
          const int c = lane + 32 * k;
          const int tok = c / C::CHUNKS, part = c % C::CHUNKS;
          const int r = __shfl_sync(0xffffffffu, row32, tok);
          const bool ok = r >= 0;
          const uint32_t off = ok ? (uint32_t)r * C::ROWB + part * 16 : 0u;
          const uint32_t dst = C::at(tok, part);
          cp_async16(kc_s + dst, kc_g + off, ok && KVQ_IN(geo, KVQ_ARRAY_K_CODES, kc_g + off, 16));
          cp_async16(vc_s + dst, vc_g + off, ok && KVQ_IN(geo, KVQ_ARRAY_V_CODES, vc_g + off, 16));
        }
      } else {
        if (lane < n) {
          if constexpr (PG) row = kch_row(geo, b, kvh, start + lane);
          else row = token_row(geo, b, kvh, start + lane);
          unmapped = row < 0;
        }
#pragma unroll
        for (int k = 0; k < C::CHUNKS; ++k) {
          const int c = lane + 32 * k;
          const int tok = c / C::CHUNKS, part = c % C::CHUNKS;
          const long long r = __shfl_sync(0xffffffffu, row, tok);
          const bool ok = r >= 0;
          const long long off = ok ? r * C::ROWB + part * 16 : 0;
          const uint32_t dst = C::at(tok, part);
          cp_async16(kc_s + dst, kc_g + off, ok && KVQ_IN(geo, KVQ_ARRAY_K_CODES, kc_g + off, 16));
          cp_async16(vc_s + dst, vc_g + off, ok && KVQ_IN(geo, KVQ_ARRAY_V_CODES, vc_g + off, 16));
        }
      }
      const unsigned bad = __ballot_sync(0xffffffffu, row < 0);
      if (lane == 0) mask_s[warp * C::STAGES + stage] = bad;
      const bool ok = row >= 0;
      const long long hoff = ok ? row * C::HDRB : 0;
      const uint32_t hdst = hd_s + lane * C::HDRB;
      if constexpr (KCH) {
        // the block's K scales then zeros, 8 channels per 16-byte chunk
        if constexpr (PG) {
          const long long hrow = kch_hdr(geo, b, kvh, (start - geo.sink) / geo.g);
          const long long hb = hrow >= 0 ? hrow * D : 0;  // unmapped: zero-filled (rows masked)
          if (lane < D / 4) {
            const int w = lane / (D / 8), c = lane % (D / 8);
            const uint8_t* hsrc = (w ? kz_g : ks_g) + (hb + c * 8) * 2;
            cp_async16(hd_s + w * 2 * D + c * 16, hsrc,
                       hrow >= 0 && KVQ_IN(geo, w ? KVQ_ARRAY_K_ZERO : KVQ_ARRAY_K_SCALE, hsrc, 16));
          }
        } else {
          const long long hb = ((((long long)b * geo.Hkv + kvh) * (geo.slots / geo.g)) +
                                (start - geo.sink) / geo.g) * D;
          if (lane < D / 4) {
            const int w = lane / (D / 8), c = lane % (D / 8);
            const uint8_t* hsrc = (w ? kz_g : ks_g) + (hb + c * 8) * 2;
            cp_async16(hd_s + w * 2 * D + c * 16, hsrc,
                       KVQ_IN(geo, w ? KVQ_ARRAY_K_ZERO : KVQ_ARRAY_K_SCALE, hsrc, 16));
          }
        }
      } else {
        cp_async_small<C::HDRB>(hdst, ks_g + hoff,
                                ok && KVQ_IN(geo, KVQ_ARRAY_K_SCALE, ks_g + hoff, C::HDRB));
        if constexpr (!SYM)
          cp_async_small<C::HDRB>(hdst + C::HDR_TILE, kz_g + hoff,
                                  ok && KVQ_IN(geo, KVQ_ARRAY_K_ZERO, kz_g + hoff, C::HDRB));
      }
      cp_async_small<C::HDRB>(hdst + C::KHB, vs_g + hoff,
                              ok && KVQ_IN(geo, KVQ_ARRAY_V_SCALE, vs_g + hoff, C::HDRB));
      if constexpr (!SYM)
        cp_async_small<C::HDRB>(hdst + C::KHB + C::HDR_TILE, vz_g + hoff,
                                ok && KVQ_IN(geo, KVQ_ARRAY_V_ZERO, vz_g + hoff, C::HDRB));
    }
    cp_async_commit();  // one group per slot, empty past the end
    return unmapped;
  };

  // ---- one tile's steps ----
  // header pass: lane = token; [token][group] fp16 -> [group][token] scratch
  auto header = [&](int stg, int buf, unsigned bad) {
    const uint8_t* hsrc = wpipe + stg * C::STAGE + 2 * C::CODE_TILE + lane * C::HDRB;
    uint32_t r[4][NG / 2];  // K scale, K zero, V scale, V zero: two halves per word
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      if (SYM && (a & 1)) continue;  // no zero rows
      if (KCH && a < 2) continue;    // no per-token K header
      const uint8_t* src = hsrc + (a < 2 ? a * C::HDR_TILE : C::KHB + (a - 2) * C::HDR_TILE);
      if constexpr (NG == 2) {
        r[a][0] = *reinterpret_cast<const uint32_t*>(src);
      } else if constexpr (NG == 4) {
        const uint2 v = *reinterpret_cast<const uint2*>(src);
        r[a][0] = v.x; r[a][1] = v.y;
      } else {
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        r[a][0] = v.x; r[a][1] = v.y; r[a][2] = v.z; r[a][3] = v.w;
      }
    }
    float2* ksz = ksz_of(buf);
    unsigned short* vs = reinterpret_cast<unsigned short*>(vsx_of(buf));
    unsigned short* vz = reinterpret_cast<unsigned short*>(vzx_of(buf));
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const int sh = (g & 1) * 16;
      if constexpr (!KCH) {
        const unsigned short uk = (unsigned short)(r[0][g / 2] >> sh);
        const unsigned short uz = SYM ? kSymZero : (unsigned short)(r[1][g / 2] >> sh);
        const float2 kv = make_float2(__half2float(__ushort_as_half(uk)) * kscale,
                                      __half2float(__ushort_as_half(uz)));
        if constexpr (TQ) ksz[lane * NG + g] = kv;   // [token][group]
        else ksz[g * C::KROW + lane] = kv;           // [group][token]
      }
      vs[g * C::VROW + lane] = (unsigned short)(r[2][g / 2] >> sh);
      vz[g * C::VROW + lane] = SYM ? kSymZero : (unsigned short)(r[3][g / 2] >> sh);
    }
    madd_of(buf)[lane] = ((bad >> lane) & 1u) ? -INFINITY : 0.f;
    if constexpr (KCH) {
      // the block's per-channel K scale and zero, reordered to [jj][kb][4]
      // (k-slot order of lane group jj) so the score pass reads its slots
      // with one 8-byte load per k-block
      if (lane < 4 * C::KB) {
        const int jj = lane & 3, kb = lane >> 2;
        int dk[4];
        slot_channels(kb, jj, dk);
        const __half* blk = reinterpret_cast<const __half*>(wpipe + stg * C::STAGE + 2 * C::CODE_TILE);
        __half* dst = reinterpret_cast<__half*>(ksz_of(buf)) + (jj * C::KB + kb) * 4;
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(pack_halves(blk[dk[0]], blk[dk[1]]), pack_halves(blk[dk[2]], blk[dk[3]]));
        // (INT4: slots 2j+8, 2j+9 meet the odd nibbles, held as 16c: their
        // zero-points are stored as 16z, exact in fp16)
        const uint32_t z23 = pack_halves(blk[D + dk[2]], blk[D + dk[3]]);
        *reinterpret_cast<uint2*>(dst + 4 * 4 * C::KB) =
            make_uint2(pack_halves(blk[D + dk[0]], blk[D + dk[1]]),
                       BITS == 4 ? h2_as_u32(__hmul2(u32_as_h2(z23), u32_as_h2(0x4C004C00u))) : z23);
      }
    }
  };

  // scores of the tile's 4 n-tiles of 8 tokens (log2 units, masked)
  auto scores = [&](int stg, int buf, unsigned bad, float (&sc)[4][2]) {
    const uint32_t kc_s = wpipe_s + stg * C::STAGE;
    const float2* ksz = ksz_of(buf);
    const float* madd = madd_of(buf);
    // A operand: q as built above, or (KCH) q times the block's per-channel
    // scale.  An fp16 product would lose 11 bits on every channel, so KCH
    // carries it as hi + lo (lo = q s - hi by one fused rounding; the pair is
    // exact to ~22 bits) and runs each score mma for both.  The zero-point
    // term -sum(A z) (and for biased codes the offset -1024 sum(A)) comes
    // from mmas against constant codes: the accumulator's start, or with
    // subnormal codes an add in the epilogue.
    uint32_t Aop[C::KB][4];
    uint32_t Alo[(KCH && !TQ) ? C::KB : 1][2];
    uint32_t Bq[(KCH && TQ) ? C::KB : 1][2];
    float kinit = 0.f, kci0 = 0.f, kci1 = 0.f;
    if constexpr (KCH && TQ) {
      // token rows: B column 0 = q s (hi), column 1 = its lo part, so one
      // mma per k-block carries both; -sum z B of both columns comes from
      // mmas with A = z (every row).  Columns 2..7 repeat the hi part: their
      // results are never read.
      const __half* sz = reinterpret_cast<const __half*>(ksz) + j * C::KB * 4;
      float ci[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb) {
        const uint2 sv = *reinterpret_cast<const uint2*>(sz + kb * 4);
        const uint2 zv = *reinterpret_cast<const uint2*>(sz + 4 * 4 * C::KB + kb * 4);
        const __half2 h01 = __hmul2(u32_as_h2(qa[kb][0]), u32_as_h2(sv.x));
        const __half2 h23 = __hmul2(u32_as_h2(qa[kb][2]), u32_as_h2(sv.y));
        const uint32_t l01 = h2_as_u32(__hfma2(u32_as_h2(qa[kb][0]), u32_as_h2(sv.x), __hneg2(h01)));
        const uint32_t l23 = h2_as_u32(__hfma2(u32_as_h2(qa[kb][2]), u32_as_h2(sv.y), __hneg2(h23)));
        Bq[kb][0] = rho == 1 ? l01 : h2_as_u32(h01);
        Bq[kb][1] = rho == 1 ? l23 : h2_as_u32(h23);
        if constexpr (!SUBK) mma16816(ci, kH1024, kH1024, kH1024, kH1024, Bq[kb][0], Bq[kb][1]);
        mma16816(ci, zv.x, zv.x, zv.y, zv.y, Bq[kb][0], Bq[kb][1]);  // zv.y: 16z for INT4
      }
      kci0 = -ci[0];  // column 2j
      kci1 = -ci[1];  // column 2j + 1
    } else if constexpr (KCH) {
      const __half* sz = reinterpret_cast<const __half*>(ksz) + j * C::KB * 4;
      float ci[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb) {
        const uint2 sv = *reinterpret_cast<const uint2*>(sz + kb * 4);
        const uint2 zv = *reinterpret_cast<const uint2*>(sz + 4 * 4 * C::KB + kb * 4);
        const __half2 h01 = __hmul2(u32_as_h2(qa[kb][0]), u32_as_h2(sv.x));
        const __half2 h23 = __hmul2(u32_as_h2(qa[kb][2]), u32_as_h2(sv.y));
        const uint32_t a01 = h2_as_u32(h01), a23 = h2_as_u32(h23);
        Alo[kb][0] = h2_as_u32(__hfma2(u32_as_h2(qa[kb][0]), u32_as_h2(sv.x), __hneg2(h01)));
        Alo[kb][1] = h2_as_u32(__hfma2(u32_as_h2(qa[kb][2]), u32_as_h2(sv.y), __hneg2(h23)));
        Aop[kb][0] = a01; Aop[kb][1] = a01; Aop[kb][2] = a23; Aop[kb][3] = a23;
        // (zv.y: slots 2j+8, 2j+9, which meet the odd nibbles held as 16c,
        // carry 16z for INT4; the header pass stored them so)
        const uint32_t b0 = rho == 0 ? kH1024 : (rho == 1 ? zv.x : 0u);
        const uint32_t b1 = rho == 0 ? kH1024 : (rho == 1 ? zv.y : 0u);
        mma16816(ci, a01, a01, a23, a23, b0, b1);
        mma16816(ci, Alo[kb][0], Alo[kb][0], Alo[kb][1], Alo[kb][1], b0, b1);
      }
      // lane (rho, 0) holds columns 0 and 1 of row rho
      kinit = __shfl_sync(0xffffffffu, -(ci[0] + ci[1]), rho << 2);
    } else {
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb)
#pragma unroll
        for (int e = 0; e < 4; ++e) Aop[kb][e] = qa[kb][e];
    }
    if constexpr (TQ) {
      float s4[4];  // this lane's tokens rho + 8i, i = 0..3
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t w[2][C::CHUNKS];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int tok = 8 * (2 * np + u) + (lane & 7);
          if constexpr (C::CHUNKS == 2) {
            ldsm_x2(kc_s + C::at(tok, (lane >> 3) & 1), w[u][0], w[u][1]);
          } else {
#pragma unroll
            for (int c4 = 0; c4 < C::CHUNKS; c4 += 4)
              ldsm_x4(kc_s + C::at(tok, c4 + (lane >> 3)), w[u][c4], w[u][c4 + 1], w[u][c4 + 2],
                      w[u][c4 + 3]);
          }
        }
        // rows: tokens rho (octet 2np) and rho + 8 (octet 2np + 1); two
        // accumulator chains (even / odd k-blocks; TQ2: the two n-tiles)
        // (axis-aware: the biased codes' offset and the zero-point term).
        // The others start at -0, which adds like +0; the build with +0
        // measured 1.5 % slower on the 7B-class step.
        const float c0 = (KCH && !SUBK) ? kci0 : -0.f, c1 = (KCH && !SUBK) ? kci1 : -0.f;
        float acc[2][4] = {{c0, c1, c0, c1}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int c = 0; c < C::CHUNKS; ++c) {
          if constexpr (BITS == 2) {
            // a chunk of 64 channels: k-blocks 4c .. 4c+3
            uint32_t h0[8], h1[8];
            crumb16_to_h2_sub(w[0][c], h0);
            crumb16_to_h2_sub(w[1][c], h1);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              mma16816(acc[i & 1], h0[2 * i], h1[2 * i], h0[2 * i + 1], h1[2 * i + 1],
                       qa[4 * c + i][0], qa[4 * c + i][2]);
          } else if constexpr (BITS == 4) {
            uint32_t h0[4], h1[4];
            if constexpr (NF) {
              nib8_to_h2_nf4_table(w[0][c], h0, nf_lut_lane);
              nib8_to_h2_nf4_table(w[1][c], h1, nf_lut_lane);
            } else {
              nib8_to_h2<NF, SUBK>(w[0][c], h0, lut);
              nib8_to_h2<NF, SUBK>(w[1][c], h1, lut);
            }
            if constexpr (TQ2) {
              const int t = qtile(2 * c);  // both k-blocks of the chunk: one group
              mma16816(acc[t], h0[0], h1[0], h0[1], h1[1], qa[2 * c][t], qa[2 * c][2 + t]);
              mma16816(acc[t], h0[2], h1[2], h0[3], h1[3], qa[2 * c + 1][t], qa[2 * c + 1][2 + t]);
            } else {
              const uint32_t b00 = KCH ? Bq[2 * c][0] : qa[2 * c][0];
              const uint32_t b01 = KCH ? Bq[2 * c][1] : qa[2 * c][2];
              const uint32_t b10 = KCH ? Bq[2 * c + 1][0] : qa[2 * c + 1][0];
              const uint32_t b11 = KCH ? Bq[2 * c + 1][1] : qa[2 * c + 1][2];
              mma16816(acc[0], h0[0], h1[0], h0[1], h1[1], b00, b01);
              mma16816(acc[1], h0[2], h1[2], h0[3], h1[3], b10, b11);
            }
          } else {
            const uint32_t a0 = byte2_to_h2_biased<0x4140, SUBK>(w[0][c]);
            const uint32_t a1 = byte2_to_h2_biased<0x4140, SUBK>(w[1][c]);
            const uint32_t a2 = byte2_to_h2_biased<0x4342, SUBK>(w[0][c]);
            const uint32_t a3 = byte2_to_h2_biased<0x4342, SUBK>(w[1][c]);
            if constexpr (TQ2) {
              const int t = qtile(c);
              mma16816(acc[t], a0, a1, a2, a3, qa[c][t], qa[c][2 + t]);
            } else {
              mma16816(acc[c & 1], a0, a1, a2, a3, KCH ? Bq[c][0] : qa[c][0], KCH ? Bq[c][1] : qa[c][2]);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          // columns 2j, 2j+1 = groups 2j, 2j+1: s (sum q c - z sum q), then
          // the groups of the other lanes of this token
          float v = 0.f;
          if constexpr (KCH) {
            // lane (rho, 0): column 0 (hi) + column 1 (lo); scales already in
            // q; subnormal codes: 2^-24 sum B c, and the zero-point term here
            const float a = (acc[0][2 * i] + acc[1][2 * i]) + (acc[0][2 * i + 1] + acc[1][2 * i + 1]);
            v = (SUBK ? fmaf(a, kSubK, kci0 + kci1) : a) * p.scale_log2;
          } else if constexpr (GP == 1) {
            if (2 * j < NG) {
              const int t = 16 * np + 8 * i + rho;
              const float4 sz = *reinterpret_cast<const float4*>(ksz + t * NG + 2 * j);
              v = sz.x * fmaf(-sz.y, qs_lo, acc[0][2 * i] + acc[1][2 * i]);
              if (2 * j + 1 < NG)
                v = fmaf(sz.z, fmaf(-sz.w, qs_hi, acc[0][2 * i + 1] + acc[1][2 * i + 1]), v);
            }
            // lane (rho, 0) must end with all groups: it is the one read below
            if constexpr (NG > 2) v += __shfl_xor_sync(0xffffffffu, v, 1);
            if constexpr (NG > 4) v += __shfl_xor_sync(0xffffffffu, v, 2);
          } else {
            // columns 2j, 2j+1 = heads 2j % GP and the next one, both of group
            // 2j / GP.  Lane j keeps one head, (j / (GP/2)) & 1 of its pair,
            // and sends the other to lane j ^ (GP/2), which holds the same
            // heads of another group and keeps the other one; GP = 2 then
            // adds the remaining groups' lanes.
            float v0 = 0.f, v1 = 0.f;
            if constexpr (TQ2) {
              // n-tile 0 holds this lane's columns for group (2j) / GP,
              // n-tile 1 for group (2j) / GP + 8 / GP
              const int t = 16 * np + 8 * i + rho;
              const float2 sz0 = ksz[t * NG + (2 * j) / GP];
              const float2 sz1 = ksz[t * NG + (2 * j) / GP + 8 / GP];
              v0 = fmaf(sz1.x, fmaf(-sz1.y, qs_lo1, acc[1][2 * i]),
                        sz0.x * fmaf(-sz0.y, qs_lo, acc[0][2 * i]));
              v1 = fmaf(sz1.x, fmaf(-sz1.y, qs_hi1, acc[1][2 * i + 1]),
                        sz0.x * fmaf(-sz0.y, qs_hi, acc[0][2 * i + 1]));
            } else if (2 * j < NG * GP) {
              const int t = 16 * np + 8 * i + rho;
              const float2 sz = ksz[t * NG + (2 * j) / GP];
              v0 = sz.x * fmaf(-sz.y, qs_lo, acc[0][2 * i] + acc[1][2 * i]);
              v1 = sz.x * fmaf(-sz.y, qs_hi, acc[0][2 * i + 1] + acc[1][2 * i + 1]);
            }
            const bool sel = (j / (GP / 2)) & 1;
            v = (sel ? v1 : v0) + __shfl_xor_sync(0xffffffffu, sel ? v0 : v1, GP / 2);
            if constexpr (GP == 2 && NG > 2) v += __shfl_xor_sync(0xffffffffu, v, 2);
          }
          s4[2 * np + i] = v;
        }
      }
      // into the softmax layout: token 8 nt + 2j + e of this lane's head
      // h_lane lives as s4[nt] in lane 4 (2j + e) + jsrc, the lane that kept
      // that head
      const int jsrc = (h_lane >> 1) + (h_lane & 1) * (GP / 2);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int ta = 8 * nt + 2 * j;
        float va = __shfl_sync(0xffffffffu, s4[nt], ((2 * j) << 2) | jsrc);
        float vb = __shfl_sync(0xffffffffu, s4[nt], ((2 * j + 1) << 2) | jsrc);
        if (bad) {  // warp-uniform
          const float2 mk = *reinterpret_cast<const float2*>(madd + ta);
          va += mk.x;
          vb += mk.y;
        }
        sc[nt][0] = va + hmask;
        sc[nt][1] = vb + hmask;
      }
    } else {
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t w[2][C::CHUNKS];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int tok = 8 * (2 * np + u) + (lane & 7);
        if constexpr (C::CHUNKS == 2) {
          ldsm_x2(kc_s + C::at(tok, (lane >> 3) & 1), w[u][0], w[u][1]);
        } else {
#pragma unroll
          for (int c4 = 0; c4 < C::CHUNKS; c4 += 4)
            ldsm_x4(kc_s + C::at(tok, c4 + (lane >> 3)), w[u][c4], w[u][c4 + 1], w[u][c4 + 2],
                    w[u][c4 + 3]);
        }
      }
      // axis-aware caches: the accumulators start at minus the biased
      // codes' offset and the zero-point term; the others at -0 (as in the
      // token-rows layout)
      float acc[2][4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        acc[u][0] = acc[u][1] = KCH ? kinit : -0.f;
        acc[u][2] = acc[u][3] = KCH ? kinit : -0.f;
      }
#pragma unroll
      for (int c = 0; c < C::CHUNKS; ++c) {
        if constexpr (BITS == 2) {
          uint32_t h0[8], h1[8];
          crumb16_to_h2_sub(w[0][c], h0);
          crumb16_to_h2_sub(w[1][c], h1);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int kb = 4 * c + i;
            mma16816(acc[0], Aop[kb][0], Aop[kb][1], Aop[kb][2], Aop[kb][3], h0[2 * i], h0[2 * i + 1]);
            mma16816(acc[1], Aop[kb][0], Aop[kb][1], Aop[kb][2], Aop[kb][3], h1[2 * i], h1[2 * i + 1]);
          }
        } else if constexpr (BITS == 4) {
          uint32_t h0[4], h1[4];
          if constexpr (NF) {
            nib8_to_h2_nf4_table(w[0][c], h0, nf_lut_lane);
            nib8_to_h2_nf4_table(w[1][c], h1, nf_lut_lane);
          } else {
            nib8_to_h2<NF, SUBK>(w[0][c], h0, lut);
            nib8_to_h2<NF, SUBK>(w[1][c], h1, lut);
          }
          mma16816(acc[0], Aop[2 * c][0], Aop[2 * c][1], Aop[2 * c][2], Aop[2 * c][3], h0[0], h0[1]);
          mma16816(acc[1], Aop[2 * c][0], Aop[2 * c][1], Aop[2 * c][2], Aop[2 * c][3], h1[0], h1[1]);
          mma16816(acc[0], Aop[2 * c + 1][0], Aop[2 * c + 1][1], Aop[2 * c + 1][2],
                   Aop[2 * c + 1][3], h0[2], h0[3]);
          mma16816(acc[1], Aop[2 * c + 1][0], Aop[2 * c + 1][1], Aop[2 * c + 1][2],
                   Aop[2 * c + 1][3], h1[2], h1[3]);
          if constexpr (KCH) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const uint32_t l01 = Alo[2 * c + e][0], l23 = Alo[2 * c + e][1];
              mma16816(acc[0], l01, l01, l23, l23, h0[2 * e], h0[2 * e + 1]);
              mma16816(acc[1], l01, l01, l23, l23, h1[2 * e], h1[2 * e + 1]);
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t h01 = byte2_to_h2_biased<0x4140, SUBK>(w[u][c]);
            const uint32_t h23 = byte2_to_h2_biased<0x4342, SUBK>(w[u][c]);
            mma16816(acc[u], Aop[c][0], Aop[c][1], Aop[c][2], Aop[c][3], h01, h23);
            if constexpr (KCH) mma16816(acc[u], Alo[c][0], Alo[c][0], Alo[c][1], Alo[c][1], h01, h23);
          }
        }
      }
      // group epilogue: row (g, h) holds sum_{d in g} q_h[d] code[d]
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int nt = 2 * np + u;
        const int ta = 8 * nt + 2 * j;
        float va, vb;
        if constexpr (KCH) {
          // rows are heads and the scales are already in A
          va = acc[u][0] * p.scale_log2;
          vb = acc[u][1] * p.scale_log2;
        } else {
          // (s*scale, z) of tokens ta and ta+1 in one 16-byte load
          const float4 szl = *reinterpret_cast<const float4*>(ksz + g_lo_c * C::KROW + ta);
          va = szl.x * fmaf(-szl.y, qs_lo, acc[u][0]);
          vb = szl.z * fmaf(-szl.w, qs_lo, acc[u][1]);
          if constexpr (C::HI) {
            const float4 szh = *reinterpret_cast<const float4*>(ksz + g_hi_c * C::KROW + ta);
            va = fmaf(szh.x, fmaf(-szh.y, qs_hi, acc[u][2]), va);
            vb = fmaf(szh.z, fmaf(-szh.w, qs_hi, acc[u][3]), vb);
          }
#pragma unroll
          for (int s2 = 0; (1 << s2) < C::NGL; ++s2) {
            va += __shfl_xor_sync(0xffffffffu, va, 4 * GP << s2);
            vb += __shfl_xor_sync(0xffffffffu, vb, 4 * GP << s2);
          }
        }
        if (bad) {  // warp-uniform: only partial tiles and unmapped pages pay for the mask
          const float2 mk = *reinterpret_cast<const float2*>(madd + ta);
          va += mk.x;
          vb += mk.y;
        }
        sc[nt][0] = va + hmask;
        sc[nt][1] = vb + hmask;
      }
    }
    }  // (group, head)-rows layout
  };

  // online softmax over the tile; pp = fp16 probabilities of this lane's tokens
  // (tk, tk+1 | tk+8, tk+9 for k-steps 0 and 1)
  auto softmax = [&](const float (&sc)[4][2], uint32_t (&pp)[4]) {
    float mt = sc[0][0];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) mt = fmaxf(mt, fmaxf(sc[nt][0], sc[nt][1]));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    // move the reference maximum only when this tile exceeds it by kSlack
    const bool need = mt > m_ref + kSlack;
    const float m_next = need ? mt : m_ref;
    if (__any_sync(0xffffffffu, need)) {
      // 0 on the first live tile; lanes that keep their reference scale by 1
      const float alpha = need ? ex2(m_ref - m_next) : 1.f;
      l_run *= alpha;
      // V columns 2j, 2j+1 (of any n-tile) belong to heads (2j) % GP, (2j+1) % GP
      const float a0 = __shfl_sync(0xffffffffu, alpha, ((2 * j) % GP) << 2);
      const float a1 = __shfl_sync(0xffffffffu, alpha, ((2 * j + 1) % GP) << 2);
#pragma unroll
      for (int m = 0; m < C::MT; ++m) {
        o[m][0] *= a0; o[m][1] *= a1; o[m][2] *= a0; o[m][3] *= a1;
      }
#pragma unroll
      for (int t = 0; t < C::NTV; ++t) {
        cz[t][0] *= a0; cz[t][1] *= a1; cz[t][2] *= a0; cz[t][3] *= a1;
      }
    }
    m_ref = m_next;
    const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
    float pr[4][2];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      pr[nt][0] = ex2(sc[nt][0] - m_use);
      pr[nt][1] = ex2(sc[nt][1] - m_use);
      l_run += pr[nt][0] + pr[nt][1];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) pp[k] = pack_h2(pr[k][0], pr[k][1]);
  };

  // weighted V of the tile: 2 k-steps of 16 tokens
  auto weighted_v = [&](int stg, int buf, const uint32_t (&pp)[4]) {
    const uint32_t vc_s = wpipe_s + stg * C::STAGE + C::CODE_TILE;
    const __half* vsx = vsx_of(buf);
    const __half* vzx = vzx_of(buf);
    // B[token][(g, h)] = p_h(token) * s_g(token); this lane's column per n-tile
    uint32_t bt[2][C::NTV][2];
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const int tk = 16 * ks + 2 * j;  // this lane's tokens: tk, tk+1, tk+8, tk+9
      const uint32_t plo = pp[2 * ks], phi = pp[2 * ks + 1];
#pragma unroll
      for (int t = 0; t < C::NTV; ++t) {
        const int g = min(gcol[t], NG - 1);
        const uint32_t slo = *reinterpret_cast<const uint32_t*>(vsx + g * C::VROW + tk);
        const uint32_t shi = *reinterpret_cast<const uint32_t*>(vsx + g * C::VROW + tk + 8);
        const bool live = gcol[t] < NG;
        bt[ks][t][0] = live ? h2_as_u32(__hmul2(u32_as_h2(plo), u32_as_h2(slo))) : 0u;
        bt[ks][t][1] = live ? h2_as_u32(__hmul2(u32_as_h2(phi), u32_as_h2(shi))) : 0u;
      }
      // zero-points: A rows = groups r, A[r][token] = z_r(token); the entries
      // with r equal to the column's group are the ones used
      const int gz = min(rho, NG - 1);
      const uint32_t zlo = rho < NG ? *reinterpret_cast<const uint32_t*>(vzx + gz * C::VROW + tk) : 0u;
      const uint32_t zhi = rho < NG ? *reinterpret_cast<const uint32_t*>(vzx + gz * C::VROW + tk + 8) : 0u;
      if constexpr (!NF) {  // NF4 has no zero-point
#pragma unroll
        for (int t = 0; t < C::NTV; ++t) mma16816(cz[t], zlo, 0u, zhi, 0u, bt[ks][t][0], bt[ks][t][1]);
      }
    }
    if constexpr (BITS <= 4) {
      // The codes are subnormals with no offset (INT4 odd nibbles 16c: their
      // rows accumulate in x16 units until the end; INT2 4^f c: rows in 4^f
      // units), or NF4 levels.
#pragma unroll
      for (int c = 0; c < C::CHUNKS; c += 2) {
        // V codes, transposed: per chunk, lo = tokens 0-7 of the k-step, hi = tokens 8-15
        uint32_t x[2][4];
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const int m = lane >> 3;
          const int tok = 16 * ks + ((m & 1) << 3) + (lane & 7);
          ldsm_x4_t(vc_s + C::at(tok, c + (m >> 1)), x[ks][0], x[ks][1], x[ks][2], x[ks][3]);
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int chunk = c + cc;
          // n-tile of the chunk's group (INT2 chunks of several groups: one n-tile)
          const int t = C::NTV == 1 ? 0 : ((chunk * C::DPC) / C::GSZ) * GP / 8;
          if constexpr (BITS == 2) {
            // m-tile 4 chunk + f: rows rho / rho + 8 = channels 64 chunk + 8 rho + f / + 4 + f
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
              uint32_t lo[8], hi[8];
              crumb16_to_h2_sub(x[ks][2 * cc], lo);
              crumb16_to_h2_sub(x[ks][2 * cc + 1], hi);
#pragma unroll
              for (int f = 0; f < 4; ++f)
                mma16816(o[4 * chunk + f], lo[f], lo[4 + f], hi[f], hi[4 + f], bt[ks][t][0], bt[ks][t][1]);
            }
          } else {
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
              uint32_t lo[4], hi[4];
              nib8_to_h2<NF, true>(x[ks][2 * cc], lo, lut);
              nib8_to_h2<NF, true>(x[ks][2 * cc + 1], hi, lut);
              // channel of lo[e] = chunk*32 + 4*rho + e; m-tile (chunk, pp) rows: e = 2pp, 2pp+1
              mma16816(o[2 * chunk], lo[0], lo[1], hi[0], hi[1], bt[ks][t][0], bt[ks][t][1]);
              mma16816(o[2 * chunk + 1], lo[2], lo[3], hi[2], hi[3], bt[ks][t][0], bt[ks][t][1]);
            }
          }
        }
      }
    } else {
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
        for (int c = 0; c < C::CHUNKS; c += 2) {
          uint32_t xlo0, xhi0, xlo1, xhi1;
          const int m = lane >> 3;
          const int tok = 16 * ks + ((m & 1) << 3) + (lane & 7);
          ldsm_x4_t(vc_s + C::at(tok, c + (m >> 1)), xlo0, xhi0, xlo1, xhi1);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const uint32_t xlo = cc ? xlo1 : xlo0, xhi = cc ? xhi1 : xhi0;
            const int chunk = c + cc;
            const int t = ((chunk * C::DPC) / C::GSZ) * GP / 8;
            const uint32_t l0 = byte2_to_h2_sub<0x4240>(xlo), l1 = byte2_to_h2_sub<0x4341>(xlo);
            const uint32_t h0 = byte2_to_h2_sub<0x4240>(xhi), h1 = byte2_to_h2_sub<0x4341>(xhi);
            mma16816(o[chunk], l0, l1, h0, h1, bt[ks][t][0], bt[ks][t][1]);
          }
        }
      }
    }
  };

  // ---- software-pipelined loop: tile i+1's scores overlap tile i's values ----
  // Tile k lives in stage k % STAGES; one commit group per tile.
#pragma unroll
  for (int s2 = 0; s2 < C::STAGES; ++s2) bt_bad |= issue(s2);

  // fused append (one warp of the owning CTA), after its first loads are in flight
  if (owner) {
    constexpr int CHV = D / 8;          // 8-channel chunks per vector
    const int which = lane / CHV;       // 0: K, 1: V, 2+: idle lanes
    const int ch = lane % CHV;
    const long long nrow = token_row(geo, b, kvh, pos_new);
    if (nrow < 0 && lane == 0 && p.status) atomicOr(p.status, KVQ_FLAG_BLOCK_TABLE);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (which < 2) {
      const uint4* src = reinterpret_cast<const uint4*>(p.new_kv[which] + ((long long)b * geo.Hkv + kvh) * D) + ch;
      if (KVQ_IN(geo, KVQ_ARRAY_K_NEW + which, src, 16)) v = __ldg(src);
    }
    Quant8 qz;
    if constexpr (NF) {
      float mid[16];  // the level midpoints, as the host computes them
#pragma unroll
      for (int i = 0; i < 15; ++i) mid[i] = __fmul_rn(__fadd_rn(p.nf4_level[i], p.nf4_level[i + 1]), 0.5f);
      mid[15] = INFINITY;
      qz = quantize8_nf4(v, C::GSZ / 8, mid);
    } else {
      qz = quantize8<BITS, SYM>(v, C::GSZ / 8);
    }
    if (which < 2 && nrow >= 0) {
      uint8_t* gcodes = const_cast<uint8_t*>(p.codes[which]) + nrow * C::ROWB + ch * BITS;
      if (KVQ_IN(geo, KVQ_ARRAY_K_CODES + which, gcodes, BITS)) {
        if constexpr (BITS == 2) *reinterpret_cast<uint16_t*>(gcodes) = (uint16_t)qz.w0;
        else if constexpr (BITS == 4) *reinterpret_cast<uint32_t*>(gcodes) = qz.w0;
        else *reinterpret_cast<uint2*>(gcodes) = make_uint2(qz.w0, qz.w1);
      }
      if (ch % (C::GSZ / 8) == 0) {
        const int g = ch / (C::GSZ / 8);
        __half* sp = const_cast<__half*>(p.scale[which]) + nrow * NG + g;
        if (KVQ_IN(geo, which ? KVQ_ARRAY_V_SCALE : KVQ_ARRAY_K_SCALE, sp, 2)) *sp = qz.s;
        if constexpr (!SYM) {
          __half* zp = const_cast<__half*>(p.zero[which]) + nrow * NG + g;
          if (KVQ_IN(geo, which ? KVQ_ARRAY_V_ZERO : KVQ_ARRAY_K_ZERO, zp, 2)) *zp = qz.z;
        }
      }
    }
    if (which < 2 && ch % (C::GSZ / 8) == 0 && qz.flags && p.status) atomicOr(p.status, qz.flags);
    // dequantized channels of this lane: (code - z) * s, exact in fp32
    const float sf = __half2float(qz.s), zf = __half2float(qz.z);
    float xh[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t code = BITS == 2 ? (qz.w0 >> (2 * k)) & 0x3u
                          : BITS == 4 ? (qz.w0 >> (4 * k)) & 0xFu
                                      : ((k < 4 ? qz.w0 : qz.w1) >> (8 * (k & 3))) & 0xFFu;
      if constexpr (NF) {
        float lv = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) lv = code == (uint32_t)i ? p.nf4_level[i] : lv;
        xh[k] = lv * sf;
      } else {
        xh[k] = ((float)code - zf) * sf;
      }
    }
    if (which == 1) {
#pragma unroll
      for (int k = 0; k < 8; ++k) tok_v[ch * 8 + k] = xh[k];
    }
    // scores q_h . k_hat over the K lanes (lanes 0 .. CHV-1), log2 units
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      float part = 0.f;
      if (which == 0 && h < G) {
#pragma unroll
        for (int k = 0; k < 8; ++k) part = fmaf(__half2float(q_s[h * D + ch * 8 + k]), xh[k], part);
      }
#pragma unroll
      for (int o2 = 1; o2 < CHV; o2 <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o2);
      if (lane == 0) tok_s[h] = h < G ? part * p.scale_log2 : -INFINITY;
    }
  }

  uint32_t pp[4] = {0u, 0u, 0u, 0u};
  if (nmine > 0) {
    cp_async_wait<C::STAGES - 1>();  // tile 0
    __syncwarp();
    const unsigned bad0 = mask_s[warp * C::STAGES];
    header(0, 0, bad0);
    __syncwarp();
    float sc[4][2];
    scores(0, 0, bad0, sc);
    softmax(sc, pp);
  }
  int stage = 0;
  // steady state, branch-free so that the two tiles' work can interleave
  for (int it = 0; it + 1 < nmine; ++it) {
    const int nstage = (stage + 1 == C::STAGES) ? 0 : stage + 1;
    float scn[4][2];
    cp_async_wait<C::STAGES - 2>();  // tile it+1
    __syncwarp();
    const unsigned badn = mask_s[warp * C::STAGES + nstage];
    header(nstage, (it + 1) & 1, badn);
    __syncwarp();
    scores(nstage, (it + 1) & 1, badn, scn);
    weighted_v(stage, it & 1, pp);
    softmax(scn, pp);
    __syncwarp();
    bt_bad |= issue(it + C::STAGES);  // into the stage tile it has just left
    stage = nstage;
  }
  if (nmine > 0) weighted_v(stage, (nmine - 1) & 1, pp);  // the last tile's values
  cp_async_wait<0>();

  // ---------------- finish this warp: l, zero-point correction ----------------
  if (bt_bad && p.status) atomicOr(p.status, KVQ_FLAG_BLOCK_TABLE);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  __syncthreads();  // every warp is done with its pipeline: reuse it for the merge

  float* red = reinterpret_cast<float*>(pipe);                 // [warps][GP][D] o
  float* ml = red + kWarps * GP * D;                            // [warps][GP][2]
#pragma unroll
  for (int m = 0; m < C::MT; ++m) {
    // rows rho / rho + 8 of m-tile m: channels d0 / d0 + d1, held in units
    // of 1 / fac (the INT4 and INT2 codes' field weights) and, for
    // subnormal codes, of 2^-24
    int d0, d1 = 1;
    float fac = 1.f;
    if constexpr (BITS == 2) {
      d0 = 64 * (m >> 2) + 8 * rho + (m & 3);
      d1 = 4;
      fac = (m & 3) == 0 ? 1.f : (m & 3) == 1 ? 0.25f : (m & 3) == 2 ? 0.0625f : 0.015625f;
    } else if constexpr (BITS == 4) {
      d0 = 32 * (m >> 1) + 4 * rho + 2 * (m & 1);
    } else {
      d0 = 16 * m + 2 * rho;
    }
    const int g = d0 / C::GSZ;  // group of the lane's rows
    const int t = g * GP / 8;
    // o[channel][(g, h)] -= cz[g][(g, h)]: row g of the correction lives in lanes 4g + j
    const float corr0 = __shfl_sync(0xffffffffu, cz[t][0], (g << 2) + j);
    const float corr1 = __shfl_sync(0xffffffffu, cz[t][1], (g << 2) + j);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = 8 * t + 2 * j + e;  // (group col / GP, head col % GP)
      const int h = col % GP;
      if (col / GP == g && h < G && warp < kWarps) {
        const float corr = e ? corr1 : corr0;
        float* dst = red + (warp * GP + h) * D;
        // INT4 (not NF4): odd rows in x16 units
        const float fe = (BITS == 2 ? fac : 1.f) * kSubV;
        const float fo = (BITS == 2 ? fac : ((BITS == 4 && !NF) ? 0.0625f : 1.f)) * kSubV;
        dst[d0] = o[m][e] * fe - corr;
        dst[d0 + d1] = o[m][2 + e] * fo - corr;
      }
    }
  }
  if (j == 0 && rho < GP && warp < kWarps) {
    ml[(warp * GP + rho) * 2] = m_ref;
    ml[(warp * GP + rho) * 2 + 1] = l_run;
  }
  // KCH: the fp16 tokens of this CTA's range (sinks, then the residual
  // window), one token per warp at a time on CUDA cores, into a second set of
  // per-warp partials
  float* red2 = ml + kWarps * GP * 2;   // [warps][GP][D]
  float* ml2 = red2 + kWarps * GP * D;  // [warps][GP][2]
  if constexpr (KCH) {
    constexpr int CPL = D / 32;         // channels per lane
    const int ns = max(0, min(t1, kS) - t0);
    const int rs = max(t0, kr0);
    const int nw = ns + max(0, t1 - rs);
    const long long wb = ((long long)b * geo.Hkv + kvh) * (geo.sink + geo.g);
    float mh[GP], lh[GP], oh[GP][CPL];
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      mh[h] = -INFINITY;
      lh[h] = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) oh[h][c] = 0.f;
    }
    // this warp's rows i = warp, warp + 4, ...: loaded WB at a time, then used
    constexpr int WB = 8;
    constexpr int WPR = CPL / 2;  // 32-bit words of a lane's channels in one row
    for (int i0 = warp; i0 < nw; i0 += kWarps * WB) {
      uint32_t kw[WB][WPR], vw[WB][WPR];
#pragma unroll
      for (int k = 0; k < WB; ++k) {
        const int i = min(i0 + k * kWarps, nw - 1);  // past the end: a row that exists, unused
        const int pos = i < ns ? t0 + i : rs + (i - ns);
        const int slot = pos < kS ? pos : geo.sink + (pos - geo.sink) % geo.g;
        // (the token this launch appends: from the input)
        const bool fresh = kch_slot >= 0 && pos == L - 1;
        const __half* kw0 = fresh ? p.new_kv[0] + ((long long)b * geo.Hkv + kvh) * D : p.window[0] + (wb + slot) * D;
        const __half* vw0 = fresh ? p.new_kv[1] + ((long long)b * geo.Hkv + kvh) * D : p.window[1] + (wb + slot) * D;
        const uint32_t* kr = reinterpret_cast<const uint32_t*>(kw0) + lane * WPR;
        const uint32_t* vr = reinterpret_cast<const uint32_t*>(vw0) + lane * WPR;
        const bool k_ok = KVQ_IN(geo, fresh ? KVQ_ARRAY_K_NEW : KVQ_ARRAY_K_WINDOW, kr, 4 * WPR);
        const bool v_ok = KVQ_IN(geo, fresh ? KVQ_ARRAY_V_NEW : KVQ_ARRAY_V_WINDOW, vr, 4 * WPR);
#pragma unroll
        for (int c = 0; c < WPR; ++c) {
          kw[k][c] = k_ok ? kr[c] : 0u;
          vw[k][c] = v_ok ? vr[c] : 0u;
        }
      }
      // scores of the batch's rows (independent, so their reductions
      // overlap), then one online-softmax update per head
      const int nb = min(WB, (nw - i0 + kWarps - 1) / kWarps);  // live rows of the batch
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        if (h >= G) continue;
        float qh[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) qh[c] = __half2float(q_s[h * D + lane * CPL + c]);
        float sc[WB];
#pragma unroll
        for (int k = 0; k < WB; ++k) {
          float part = 0.f;
#pragma unroll
          for (int c = 0; c < WPR; ++c) {
            const float2 kx = __half22float2(u32_as_h2(kw[k][c]));
            part = fmaf(qh[2 * c], kx.x, part);
            part = fmaf(qh[2 * c + 1], kx.y, part);
          }
          sc[k] = part;
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) {
#pragma unroll
          for (int k = 0; k < WB; ++k) sc[k] += __shfl_xor_sync(0xffffffffu, sc[k], o2);
        }
        float mx = mh[h];
#pragma unroll
        for (int k = 0; k < WB; ++k) {
          sc[k] = k < nb ? sc[k] * p.scale_log2 : -INFINITY;
          mx = fmaxf(mx, sc[k]);
        }
        const float a = mh[h] == -INFINITY ? 0.f : ex2(mh[h] - mx);
        lh[h] *= a;
#pragma unroll
        for (int c = 0; c < CPL; ++c) oh[h][c] *= a;
#pragma unroll
        for (int k = 0; k < WB; ++k) {
          const float e = ex2(sc[k] - mx);  // 0 for the rows past the end
          lh[h] += e;
#pragma unroll
          for (int c = 0; c < WPR; ++c) {
            const float2 vx = __half22float2(u32_as_h2(vw[k][c]));
            oh[h][2 * c] = fmaf(e, vx.x, oh[h][2 * c]);
            oh[h][2 * c + 1] = fmaf(e, vx.y, oh[h][2 * c + 1]);
          }
        }
        mh[h] = mx;
      }
    }
    if (kch_slot >= 0 && warp == 0 && lane < D / 4) {  // the appended token's fp16 slot
      const int which = lane / (D / 8), ch = lane % (D / 8);
      const long long bh = (long long)b * geo.Hkv + kvh;
      uint4* to = reinterpret_cast<uint4*>(const_cast<__half*>(p.window[which]) + (bh * (geo.sink + geo.g) + kch_slot) * D) + ch;
      const uint4* from = reinterpret_cast<const uint4*>(p.new_kv[which] + bh * D) + ch;
      if (KVQ_IN(geo, KVQ_ARRAY_K_NEW + which, from, 16) && KVQ_IN(geo, KVQ_ARRAY_K_WINDOW + which, to, 16))
        *to = *from;
    }
#pragma unroll
    for (int h = 0; h < GP; ++h) {
#pragma unroll
      for (int c = 0; c < CPL; ++c) red2[(warp * GP + h) * D + lane * CPL + c] = oh[h][c];
      if (lane == 0) {
        ml2[(warp * GP + h) * 2] = mh[h];
        ml2[(warp * GP + h) * 2 + 1] = lh[h];
      }
    }
  }
  __syncthreads();

  const long long hq0 = (long long)b * p.Hq + (long long)kvh * G;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, d = i - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) M = fmaxf(M, ml[(w2 * GP + h) * 2]);
    if constexpr (KCH) {
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) M = fmaxf(M, ml2[(w2 * GP + h) * 2]);
    }
    const float ms = owner_cta ? tok_s[h] : -INFINITY;  // the appended token's partial
    M = fmaxf(M, ms);
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) {
        const float f = exp2f(ml[(w2 * GP + h) * 2] - M);
        num = fmaf(f, red[(w2 * GP + h) * D + d], num);
        den = fmaf(f, ml[(w2 * GP + h) * 2 + 1], den);
      }
      if constexpr (KCH) {
#pragma unroll
        for (int w2 = 0; w2 < kWarps; ++w2) {
          const float f = exp2f(ml2[(w2 * GP + h) * 2] - M);
          num = fmaf(f, red2[(w2 * GP + h) * D + d], num);
          den = fmaf(f, ml2[(w2 * GP + h) * 2 + 1], den);
        }
      }
      if (owner_cta) {
        const float f = exp2f(ms - M);
        num = fmaf(f, tok_v[d], num);
        den += f;
      }
    }
    if (p.splits == 1) {
      if (KVQ_IN(geo, KVQ_ARRAY_OUT, p.out + hq0 * D + i, 2))
        p.out[hq0 * D + i] = __float2half_rn(den > 0.f ? num / den : 0.f);
    } else {
      float* w = p.ws_o + ((hq0 + h) * p.splits + split) * D + d;
      if (KVQ_IN(geo, KVQ_ARRAY_WORKSPACE, w, 4)) *w = num;
      if (d == 0) {
        float* mlo = p.ws_ml + ((hq0 + h) * p.splits + split) * 2;
        if (KVQ_IN(geo, KVQ_ARRAY_WORKSPACE, mlo, 8)) {
          mlo[0] = M;
          mlo[1] = den;
        }
      }
    }
  }
}

// Launches the instantiation, or with ctas_per_sm != nullptr only reports
// how many of its CTAs fit on one SM.
template <int BITS, int D, int NG, int GP, bool SYM, bool KCH = false, bool NF = false,
          bool PG = false>
cudaError_t launch_fast_inst(const DecodeParams& p, cudaStream_t stream, int* ctas_per_sm) {
  const size_t smem = NF ? nf_lut_offset<BITS, D, NG, GP, KCH>() + kNfLutBytes
                          : fast_smem_bytes<BITS, D, NG, GP, KCH>();
  static KernelSetup setup;  // the shared-memory attribute and occupancy, once per device
  const cudaError_t e = setup_kernel(decode_fast_kernel<BITS, D, NG, GP, SYM, KCH, NF, PG>, setup,
                                     Cfg<BITS, D, NG, GP, KCH>::THREADS, smem, ctas_per_sm);
  if (e != cudaSuccess || ctas_per_sm) return e;
  // programmatic stream serialization: this launch may overlap the tail of the
  // previous kernel in the stream; the kernel waits for it before using any
  // caller data
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.geom.Hkv, p.batch);
  // the append warp only runs in the fused step
  cfg.blockDim = dim3(p.lens_before != nullptr ? Cfg<BITS, D, NG, GP, KCH>::THREADS : kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_fast_kernel<BITS, D, NG, GP, SYM, KCH, NF, PG>, p);
}

}  // namespace fast
}  // namespace kvq
