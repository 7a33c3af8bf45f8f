// k_gemm_tc.cu -- linear_bf16 on the 5th-generation tensor cores ("deepseek_v41_ref::attn"
// precision contract: bf16 operands, f32 accumulation, bf16 result): y[m][n] = sum_k x[m][k] W[n][k].
//
// Orientation: the weight is the MMA's A operand (M = 128 output features per tile) and the
// activations its B operand (N = BN tokens per tile, 16..256), so a decode step with a few dozen
// tokens still issues full 128-row MMAs while the weights stream from HBM exactly once.
// Both operands are K-major and arrive by TMA in 64-element (128-byte) swizzled slices; the
// accumulator lives in TMEM (two BN-column buffers so the epilogue of one tile overlaps the MMAs of
// the next).
//
// Work split: the (tile, 64-wide k-slice) units of up to four independent problems (several weights
// applied to the same activations, or the groups of the block-diagonal wo_a) are laid end to end
// and divided evenly over a persistent grid of at most one CTA per SM ("Stream-K"; a weight-streaming
// launch takes a slightly smaller grid when one of at least 80% of the SMs gives every CTA whole
// tiles, or equal fractions of one, which removes or evens out the fixups).  A tile whose k-range
// spans several CTAs is finished by whichever of them arrives last: each writes its f32 partial to
// the workspace, bumps the tile's arrival counter, and the last one sums the partials in CTA order
// (deterministic) and writes the bf16 result.  No CTA ever waits for another.
//
// Prefill-sized launches (many token tiles, activations far beyond L2) run k_gemm_tc_waves instead:
// whole tiles in data-parallel waves (CTA c takes tiles c, c + G, ...), so that the tiles in flight
// together are consecutive ones whose operands share L2, then Stream-K over the last partial wave.
// Launches of 2048 tokens or more on bf16 weights go one step further, to k_gemm_tc_pairs: clusters
// of two CTAs on neighbouring weight tiles of one 256-token tile, each copying half of the token
// tile and multicasting it into both (a third less L2 operand traffic a CTA).
// L2 policies follow the reuse: weights read by one token tile only stream past evict-first,
// activations small next to L2 stay evict-last, everything else is normal.
//
// Warp roles (192 threads): warps 0-3 epilogue (TMEM lane quadrant = warp), warp 4 TMA producer,
// warp 5 TMEM allocation + MMA issue.  Every mbarrier wait is time-bounded; a timeout raises the
// device status word and the CTA drains its copies and MMAs, frees TMEM and exits.
#include <mutex>

#include "csa_internal.cuh"
#include "tc_ptx.cuh"

#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace csa {

namespace gemm {

constexpr int kMaxProblems = 4;
constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle atom of K
#ifndef CSA_GEMM_ATOMS
#define CSA_GEMM_ATOMS 1
#endif
constexpr int ATOMS = CSA_GEMM_ATOMS;  // k-slices per pipeline stage: ATOMS * 128 contiguous bytes per weight row
constexpr int kThreads = 192;
// fp8 weights: four more warps (6-9) expand the weights beside the epilogue warps
constexpr int kThreadsF8 = 320;
template <bool kF8>
constexpr int threads_of() { return kF8 ? kThreadsF8 : kThreads; }
constexpr int kCounterInts = 65536;            // arrival counters at the head of the workspace
constexpr size_t kCounterBytes = kCounterInts * sizeof(int);
constexpr int kMaxContrib = 320;  // >= grid + 1 for any grid of one CTA per SM
// activations above this size (well beyond the 126 MiB L2 once the weights stream beside them) are
// read in whole-tile waves; smaller ones stay in L2 under Stream-K's contiguous ranges, which
// measured faster there
constexpr size_t kWaveActBytes = (size_t)96 << 20;

struct Problem {
  CUtensorMap tmA;  // W [groups*N rows][Kg] bf16, box {64, 128}
  CUtensorMap tmB;  // x [M rows][groups*Kg] bf16, box {64, BN}
  bf16 *y;
  int ldy, N, M, groups, Kg, kblocks, tiles_n, tiles_m, tiles, unit_begin, tile_begin;
  float *part;  // split-K mode
  int ldp;
  // L2 policies of the two operands' copies: 0 evict-first, 1 normal, 2 evict-last
  int pol_a, pol_b;
  // fp8 weights (kernels instantiated with kF8): tmA maps the e4m3 codes (uint8 [groups*N][Kg], box
  // {64, 128}, unswizzled), with one f32 scale per 128 x 128 tile at scale[(row/128) * ld_scale + k/128]
  const float *scale;
  int ld_scale;
};

struct Params {
  Problem prob[kMaxProblems];
  int nprob, total_units, total_tiles, BN, stages;
  int cstages;  // kF8: stages of the converted (bf16) weight ring
  int split_S;  // > 0: split-K mode, CTA c = (tile c / S, k-range c % S), partials out, no fixup
  // data-parallel waves: CTA c first takes the whole tiles c, c + G, ... (dp_waves of them; tiles
  // [0, dp_waves G) in all), then its Stream-K share of the units from sk_unit0 on
  int dp_waves, sk_unit0;
  // k_gemm_tc_pairs: the pair tiles [pt_begin, pt_begin + pt_count) of the launch; ksplit > 1: each
  // split over ksplit equal k-ranges, the f32 partial sums to tail_part [ksplit][pt_count][256][256]
  int pt_begin, pt_count, ksplit;
  float *tail_part;
  int early_dependents;  // let a programmatic dependent launch once every CTA here has started
  // launched as a programmatic dependent of the kernel before it (k_gemm_tc only): the producer
  // copies the weights of its first stages, then waits for that kernel, then copies their activations
  int pdl;
  float *partials;  // [grid][2][BM][BN]
  int *counters;    // [total_tiles]
  int *status;
};

struct Unit {
  int p, tile, kb;
};

// Failure-detection test hook of this device (csa_debug_stall): while nonzero, the MMA issuer of
// every CTA first waits -- giving up after this many nanoseconds -- for a phase of its drain barrier
// that nothing completes before its own final commit, so that the CTA takes its timeout path for
// certain: the other roles see the abort flag, the producer lets its copies in flight land, the
// status word records the timeout.
__device__ unsigned long long g_stall_ns = 0ull;
__device__ __forceinline__ uint64_t stall_ns() { return *const_cast<volatile unsigned long long *>(&g_stall_ns); }

__device__ __forceinline__ Unit decode_unit(const Params &P, int u) {
  int p = 0;
  while (p + 1 < P.nprob && u >= P.prob[p + 1].unit_begin) ++p;
  const int local = u - P.prob[p].unit_begin;
  return Unit{p, local / P.prob[p].kblocks, local % P.prob[p].kblocks};
}

__device__ __forceinline__ int64_t cta_start(int64_t c, int64_t U, int64_t G) { return c * U / G; }
__device__ __forceinline__ int64_t unit_owner(int64_t v, int64_t U, int64_t G) { return ((v + 1) * G - 1) / U; }

// Units [ub, ue) of segment s of this CTA: whole tile blockIdx.x + s G for s < dp_waves, then the
// Stream-K share of the rest (split-K mode: the one k-range of the CTA's tile).
template <bool kWaves>
__device__ __forceinline__ void seg_range(const Params &P, int s, int &ub, int &ue) {
  const int64_t G = gridDim.x;
  if (!kWaves && P.split_S > 0) {
    const int tg = blockIdx.x / P.split_S, sp = blockIdx.x % P.split_S;
    int p = 0;
    while (p + 1 < P.nprob && tg >= P.prob[p + 1].tile_begin) ++p;
    const int kps = P.prob[p].kblocks / P.split_S;
    ub = P.prob[p].unit_begin + (tg - P.prob[p].tile_begin) * P.prob[p].kblocks + sp * kps;
    ue = ub + kps;
  } else if (kWaves && s < P.dp_waves) {
    const int t = blockIdx.x + s * (int)G;
    int p = 0;
    while (p + 1 < P.nprob && t >= P.prob[p + 1].tile_begin) ++p;
    ub = P.prob[p].unit_begin + (t - P.prob[p].tile_begin) * P.prob[p].kblocks;
    ue = ub + P.prob[p].kblocks;
  } else {
    const int sk0 = kWaves ? P.sk_unit0 : 0;  // (no waves: the whole launch is Stream-K)
    const int64_t Usk = P.total_units - sk0;
    ub = sk0 + (int)cta_start(blockIdx.x, Usk, G);
    ue = sk0 + (int)cta_start(blockIdx.x + 1, Usk, G);
  }
}

// fp8 weights: one stage's e4m3 codes (128 rows x 128 codes, row-major, 128 bytes a row: two 64-wide
// k-slices) are expanded into the two bf16 operands the MMA reads (each 128 rows x 128 bytes, 128-byte
// swizzle: 16-byte chunk c of row r at r * 128 + ((c ^ (r % 8)) << 4)), each value times its tile's
// scale: w = bf16(f32(e4m3) * scale) with one f32 rounding of the product (exact e4m3 -> f32), the
// bf16 weight the converter of the pages' checkpoint produces.  Two groups of 128 threads share a
// stage: group IT0 / 4 takes the 16-byte code chunks q = it * 128 + t for it = IT0 .. IT0 + 3
// (contiguous per warp; chunk q is row q / 8, codes 16 (q % 8) ..).  row0 = the tile's first weight
// row; rows at or past nrows (the ragged end) get scale 0.
// atomicAdd with acquire-release semantics at gpu scope (returns the old value)
__device__ __forceinline__ int atom_add_acq_rel_gpu(int *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// The scale of a stage whose 128 rows lie in one 128-row scale block (every aligned tile), read ahead
// of the stage's wait so that its latency hides behind the copy; 0 for a tile across two blocks.
__device__ __forceinline__ float fp8_stage_scale(const float *scale, int ld_scale, int row0, int nrows, int kcol) {
  const bool one = (row0 & 127) == 0 && row0 + 128 <= nrows;
  return one ? __ldg(scale + (int64_t)(row0 >> 7) * ld_scale + kcol) : 0.f;
}

template <int IT0>
__device__ __forceinline__ void fp8_expand_half(const uint8_t *raw, uint8_t *dst, const float *scale, int ld_scale,
                                                int row0, int nrows, int kcol, int t, float sc0) {
  const bool one = (row0 & 127) == 0 && row0 + 128 <= nrows;
#pragma unroll
  for (int it = IT0; it < IT0 + 4; ++it) {
    const int q = it * 128 + t, r = q >> 3, slice = (q >> 2) & 1, part = q & 3;
    const int gr = row0 + r;
    const float sc = one ? sc0 : (gr < nrows ? __ldg(scale + (int64_t)(gr >> 7) * ld_scale + kcol) : 0.f);
    const uint4 v = *reinterpret_cast<const uint4 *>(raw + q * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)((w[k] >> (16 * h)) & 0xffffu), __NV_E4M3);
        const float2 f = __half22float2(__half2(hr));
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(f.x, sc), __fmul_rn(f.y, sc));
        o[2 * k + h] = *reinterpret_cast<const uint32_t *>(&b2);
      }
    }
    uint8_t *rp = dst + slice * (BM * BK * 2) + r * 128;
    *reinterpret_cast<uint4 *>(rp + (((2 * part) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4 *>(rp + (((2 * part + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// The product for few token tiles (decode) and split-K: each CTA one contiguous Stream-K range of
// units (or one k-range of a tile).
template <bool kF8>
__global__ void __launch_bounds__(threads_of<kF8>(), kF8 ? 1 : 2) k_gemm_tc(const __grid_constant__ Params P) {
  // a programmatic dependent after this launch that reads its output only after its dependency wait
  // (the fused indexer after proj qr) may start on the SMs this grid leaves
  if (P.early_dependents) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const int S = P.stages, BN = P.BN;
  const uint32_t a_atom = BM * BK * 2, b_atom = (uint32_t)BN * BK * 2;
  // k-slices a stage holds: fp8 weights take two, so that each code row of a stage is 128 bytes
  constexpr int KS = kF8 ? 2 : ATOMS;
  const uint32_t a_bytes = KS * a_atom, b_bytes = KS * b_atom;
  // kF8: a stage holds the fp8 codes (a8_bytes: 128 rows x 128 codes) and B; the expanded bf16
  // weights go to a ring of SC slots of a_bytes after the stages
  constexpr uint32_t a8_bytes = BM * BK * KS;
  const uint32_t a_in = kF8 ? a8_bytes : a_bytes;  // bytes of A in a stage
  const uint32_t stage_bytes = a_in + b_bytes;
  const int SC = kF8 ? P.cstages : 0;
  uint8_t *conv = smem + S * stage_bytes;
  uint64_t *full = reinterpret_cast<uint64_t *>(conv + SC * a_bytes);
  uint64_t *empty = full + S;
  uint64_t *cfull = empty + S;    // kF8 [SC]: expanded weights ready (the 128 converter threads)
  uint64_t *cempty = cfull + SC;  // kF8 [SC]: slot read by its MMAs
  uint64_t *accf = cempty + SC;   // [2]
  uint64_t *acce = accf + 2;   // [2]
  uint64_t *drain = acce + 2;
  uint64_t *epi = drain + 1;  // the 128 epilogue threads' own barrier
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(epi + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_last = const_cast<int *>(abort_flag) + 1;
  int *cslot = s_last + 1;  // [kMaxContrib] partial slots of a tile's contributors, in CTA order

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t U = P.total_units, G = gridDim.x;
  int u0, u1;
  if (P.split_S > 0) {
    const int tg = blockIdx.x / P.split_S, sp = blockIdx.x % P.split_S;
    int p = 0;
    while (p + 1 < P.nprob && tg >= P.prob[p + 1].tile_begin) ++p;
    const int kps = P.prob[p].kblocks / P.split_S;
    u0 = P.prob[p].unit_begin + (tg - P.prob[p].tile_begin) * P.prob[p].kblocks + sp * kps;
    u1 = u0 + kps;
  } else {
    u0 = (int)cta_start(blockIdx.x, U, G);
    u1 = (int)cta_start(blockIdx.x + 1, U, G);
  }
  if (u0 >= u1) {
    if (P.pdl) asm volatile("griddepcontrol.wait;" ::: "memory");  // (this grid ends after the one before)
    return;
  }
  const uint32_t tmem_cols = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int c = 0; c < SC; ++c) {
      tc::mbar_init(&cfull[c], 256);  // both converter groups
      tc::mbar_init(&cempty[c], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], 128);
    }
    tc::mbar_init(drain, 1);
    tc::mbar_init(epi, 128);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 5) tc::tmem_alloc(tmem_slot, tmem_cols);
  if (warp == 4 && lane == 0) {
    for (int p = 0; p < P.nprob; ++p) {
      tc::prefetch_tmap(&P.prob[p].tmA);
      tc::prefetch_tmap(&P.prob[p].tmB);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 4) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_first = tc::policy_evict_first(), pol_normal = tc::policy_evict_normal(),
                     pol_last = tc::policy_evict_last();
      auto pol = [&](int sel) { return sel == 0 ? pol_first : (sel == 1 ? pol_normal : pol_last); };
      const uint64_t pol_w = pol(P.prob[0].pol_a), pol_x = pol(P.prob[0].pol_b);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      // the unit's coordinates, decoded once and then advanced without divisions (this loop paces
      // the copies)
      Unit un = decode_unit(P, u0);
      const Problem *pr = &P.prob[un.p];
      int tm = un.tile % pr->tiles_m, tn = (un.tile / pr->tiles_m) % pr->tiles_n;
      int g = un.tile / (pr->tiles_m * pr->tiles_n);
      // the copies of one unit into a stage: its weights (A) and / or its activations (B)
      auto load = [&](int st, bool a_part, bool b_part) {
        uint8_t *sa = smem + st * stage_bytes;
#pragma unroll
        for (int a = 0; a < KS; ++a) {
          const int k0 = (un.kb * KS + a) * BK;
          if (a_part && (!kF8 || a == 0))  // (fp8: one box of 128 codes a row covers both slices)
            tc::tma_load_2d(sa + a * a_atom, &pr->tmA, &full[st], k0, g * pr->N + tn * BM, pol_w);
          if (b_part) tc::tma_load_2d(sa + a_in + a * b_atom, &pr->tmB, &full[st], g * pr->Kg + k0, tm * BN, pol_x);
        }
      };
      auto advance = [&]() {
        if (++un.kb == pr->kblocks) {  // next tile: token tile fastest, then weight tile, then group
          un.kb = 0;
          if (++un.tile == pr->tiles) {
            un.tile = 0;
            tm = tn = g = 0;
            if (++un.p < P.nprob) pr = &P.prob[un.p];
          } else if (++tm == pr->tiles_m) {
            tm = 0;
            if (++tn == pr->tiles_n) {
              tn = 0;
              ++g;
            }
          }
        }
      };
      int u = u0;
      if (P.pdl) {
        // the weights of the first stages stream in while the kernel before finishes; its output
        // (the activations) is copied only after the dependency wait
        const Unit un0 = un;
        const Problem *pr0 = pr;
        const int tm0 = tm, tn0 = tn, g0 = g;
        const int npre = min(S, u1 - u0);
        for (int i = 0; i < npre; ++i) {
          tc::mbar_expect_tx(&full[i], stage_bytes);
          load(i, true, false);
          advance();
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        un = un0;
        pr = pr0;
        tm = tm0;
        tn = tn0;
        g = g0;
        for (int i = 0; i < npre; ++i) {
          load(i, false, true);
          advance();
        }
        issued = npre;
        u = u0 + npre;
        stage = npre == S ? 0 : npre;
        phase = npre == S ? 1u : 0u;
      }
      for (; u < u1; ++u) {
        if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag)) break;
        tc::mbar_expect_tx(&full[stage], stage_bytes);
        load(stage, true, true);
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
        advance();
      }
      // let every copy this CTA issued land before the CTA can exit
      for (int i = issued - S > 0 ? issued - S : 0; i < issued; ++i) {
        uint64_t *b = &full[i % S];
        const uint32_t par = (uint32_t)((i / S) & 1);
        const uint64_t t0 = tc::global_ns();
        while (!tc::mbar_try_wait(b, par) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int cst = 0;  // kF8: slot of the expanded-weight ring, and its phase
      uint32_t cph = 0;
      int used[2] = {0, 0};
      int buf = 0;
      int u = u0;
      bool ok = true;
      if (const uint64_t st = stall_ns()) ok = tc::mbar_wait(drain, 0, abort_flag, st);  // test hook
      while (u < u1 && ok) {
        const Unit un = decode_unit(P, u);
        const Problem &pr = P.prob[un.p];
        const int seg_end = min(u1, pr.unit_begin + (un.tile + 1) * pr.kblocks);
        if (!tc::mbar_wait(&acce[buf], (uint32_t)(used[buf] & 1) ^ 1u, abort_flag)) break;
        tc::tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * BN);
        bool first = true;
        for (; u < seg_end; ++u) {
          if (!tc::mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          if constexpr (kF8) {  // the expanded weights of this unit
            if (!tc::mbar_wait(&cfull[cst], cph, abort_flag)) {
              ok = false;
              break;
            }
          }
          tc::tc_fence_after();
          const uint32_t sa = tc::smem_u32(smem + stage * stage_bytes);
          const uint32_t sa_w = kF8 ? tc::smem_u32(conv + cst * a_bytes) : sa;
#pragma unroll
          for (int a = 0; a < KS; ++a) {
            const uint64_t ad = tc::sdesc_sw128(sa_w + a * a_atom, 16, 1024);
            const uint64_t bd = tc::sdesc_sw128(sa + a_in + a * b_atom, 16, 1024);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              tc::mma_bf16(d, ad + 2ull * k, bd + 2ull * k, idesc, (first && a == 0 && k == 0) ? 0u : 1u);
          }
          first = false;
          tc::mma_commit(&empty[stage]);
          if constexpr (kF8) {
            tc::mma_commit(&cempty[cst]);
            if (++cst == SC) {
              cst = 0;
              cph ^= 1u;
            }
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit(&accf[buf]);
        ++used[buf];
        buf ^= 1;
      }
      // every MMA issued has completed once this arrives
      tc::mma_commit(drain);
      const uint64_t t0 = tc::global_ns();
      while (!tc::mbar_try_wait(drain, 0) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
      }
    }
  } else if (kF8 && warp >= 6) {
    // ---------------------------------------------------------------- fp8 expansion (warps 6-9)
    // the second half of every stage's codes, in unit order, beside the epilogue warps' first half
    const int t = threadIdx.x - 192;
    int rst = 0, cst = 0;
    uint32_t rph = 0, cph = 0;
    for (int sg = 0; sg < 1; ++sg) {
      int ub, ue;
      ub = u0;
      ue = u1;
      bool okc = true;
      for (int v = ub; v < ue; ++v) {
        const Unit un = decode_unit(P, v);
        const Problem &pr = P.prob[un.p];
        const int rest = un.tile / pr.tiles_m, tn = rest % pr.tiles_n, g = rest / pr.tiles_n;
        const int row0 = g * pr.N + tn * BM, kcol = un.kb;
        const float sc0 = fp8_stage_scale(pr.scale, pr.ld_scale, row0, pr.N * pr.groups, kcol);
        if (!(okc = tc::mbar_wait(&full[rst], rph, abort_flag))) break;
        if (!(okc = tc::mbar_wait(&cempty[cst], cph ^ 1u, abort_flag))) break;
        fp8_expand_half<4>(smem + rst * stage_bytes, conv + cst * a_bytes, pr.scale, pr.ld_scale, row0,
                           pr.N * pr.groups, kcol, t, sc0);
        fence_proxy_async_smem();
        tc::mbar_arrive(&cfull[cst]);
        if (++rst == S) {
          rst = 0;
          rph ^= 1u;
        }
        if (++cst == SC) {
          cst = 0;
          cph ^= 1u;
        }
      }
      if (!okc) break;
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- epilogue (warps 0-3)
    const int row = warp * 32 + lane;  // feature within the tile
    int done[2] = {0, 0};
    uint32_t epi_uses = 0;
    auto epi_sync = [&]() -> bool {
      tc::mbar_arrive(epi);
      return tc::mbar_wait(epi, (epi_uses++) & 1u, abort_flag);
    };
    // kF8: expand the weights of units [v0, v1) of one tile (first k-slice kb0, weight rows from
    // row0), in unit order, into the expanded-weight ring
    int rst = 0, cst = 0;
    uint32_t rph = 0, cph = 0;
    auto convert_units = [&](int v0, int v1, const Problem &pr, int row0, int kb0) -> bool {
      for (int v = v0; v < v1; ++v) {
        const int kcol = kb0 + v - v0;  // (a unit is one 128-wide scale column)
        const float sc0 = fp8_stage_scale(pr.scale, pr.ld_scale, row0, pr.N * pr.groups, kcol);
        if (!tc::mbar_wait(&full[rst], rph, abort_flag)) return false;
        if (!tc::mbar_wait(&cempty[cst], cph ^ 1u, abort_flag)) return false;
        fp8_expand_half<0>(smem + rst * stage_bytes, conv + cst * a_bytes, pr.scale, pr.ld_scale, row0,
                           pr.N * pr.groups, kcol, threadIdx.x, sc0);
        fence_proxy_async_smem();
        tc::mbar_arrive(&cfull[cst]);
        if (++rst == S) {
          rst = 0;
          rph ^= 1u;
        }
        if (++cst == SC) {
          cst = 0;
          cph ^= 1u;
        }
      }
      return true;
    };
    int buf = 0;
    int u = u0;
    const int first_tile_global = [&] {
      const Unit f = decode_unit(P, u0);
      return P.prob[f.p].tile_begin + f.tile;
    }();
    while (u < u1) {
      const Unit un = decode_unit(P, u);
      const Problem &pr = P.prob[un.p];
      const int tile_u0 = pr.unit_begin + un.tile * pr.kblocks, tile_u1 = tile_u0 + pr.kblocks;
      const int seg_end = min(u1, tile_u1);
      const bool whole = (u == tile_u0) && (seg_end == tile_u1);
      const int tm = un.tile % pr.tiles_m, rest = un.tile / pr.tiles_m;
      const int tn = rest % pr.tiles_n, g = rest / pr.tiles_n;
      const int f = tn * BM + row;
      const bool f_ok = f < pr.N;
      bf16 *ycol = pr.y + (int64_t)g * pr.N + f;
      const int gtile = pr.tile_begin + un.tile;
      if constexpr (kF8) {
        if (!convert_units(u, seg_end, pr, g * pr.N + tn * BM, un.kb)) break;
      }
      if (!tc::mbar_wait(&accf[buf], (uint32_t)(done[buf] & 1), abort_flag)) break;
      tc::tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * BN);
      if (P.split_S > 0) {
        // split-K: this CTA's partial sum for (tile, k-range) as f32, coalesced over features
        const int sp = blockIdx.x % P.split_S;
        float *pcol = pr.part + (int64_t)g * pr.N + f;
        for (int c0 = 0; c0 < BN; c0 += 16) {
          uint32_t r[16];
          tc::tmem_ld16(taddr + (uint32_t)c0, r);
          tc::tmem_ld_wait();
          if (f_ok) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j = tm * BN + c0 + i;
              if (j < pr.M) pcol[((int64_t)sp * pr.M + j) * pr.ldp] = __uint_as_float(r[i]);
            }
          }
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&acce[buf]);
        ++done[buf];
        buf ^= 1;
        u = seg_end;
        continue;
      }
      const int slot = (int)blockIdx.x * 2 + (gtile == first_tile_global ? 0 : 1);
      // partial tile layout: 4-column groups, the group's 128 rows contiguous (row r, columns 4c..4c+3
      // at (c * BM + r) * 4), so that a warp's 16-byte stores and loads cover 512 contiguous bytes
      float *mine = P.partials + (size_t)slot * BM * BN;
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t r[16];
        tc::tmem_ld16(taddr + (uint32_t)c0, r);
        tc::tmem_ld_wait();
        if (whole) {
          if (f_ok) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j = tm * BN + c0 + i;
              if (j < pr.M) ycol[(int64_t)j * pr.ldy] = __float2bfloat16_rn(__uint_as_float(r[i]));
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4 *>(mine + ((size_t)((c0 + i) >> 2) * BM + row) * 4) =
                make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]), __uint_as_float(r[i + 2]),
                            __uint_as_float(r[i + 3]));
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&acce[buf]);
      ++done[buf];
      buf ^= 1;
      if (!whole) {
        // Stream-K fixup: the last contributor of this tile sums the partials in CTA order.  The
        // partials are published by one gpu-scope release after the CTA's barrier (the barrier
        // orders every thread's stores before it), and the last arriver's acquire on the same
        // counter, passed on by the barrier after it, orders its reads after the others' stores.
        if (!epi_sync()) break;
        const int64_t c_first = unit_owner(tile_u0, U, G), c_last = unit_owner(tile_u1 - 1, U, G);
        if (threadIdx.x == 0) {
          const int old = atom_add_acq_rel_gpu(&P.counters[gtile], 1);
          *s_last = (old == (int)(c_last - c_first)) ? 1 : 0;
        }
        if (!epi_sync()) break;
        if (*s_last) {
          const int nc = (int)(c_last - c_first + 1);
          for (int i = threadIdx.x; i < nc; i += 128) {
            const int64_t c = c_first + i;
            const Unit f0 = decode_unit(P, (int)cta_start(c, U, G));
            cslot[i] = (int)c * 2 + (gtile == P.prob[f0.p].tile_begin + f0.tile ? 0 : 1);
          }
          if (!epi_sync()) break;
          // sum the contributors' rows in CTA order, four contributors' 16-column chunks in flight
          const float *base = P.partials + (size_t)row * 4;
          for (int c0 = 0; c0 < BN; c0 += 16) {
            float a[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) a[i] = 0.f;
            for (int i = 0; i < nc; i += 4) {
              float4 v[4][4];
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (i + q < nc) {
                  const float *src = base + (size_t)cslot[i + q] * BM * BN + (size_t)(c0 >> 2) * BM * 4;
#pragma unroll
                  for (int k = 0; k < 4; ++k) v[q][k] = __ldcg(reinterpret_cast<const float4 *>(src + (size_t)k * BM * 4));
                }
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (i + q < nc) {
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    a[4 * k] += v[q][k].x;
                    a[4 * k + 1] += v[q][k].y;
                    a[4 * k + 2] += v[q][k].z;
                    a[4 * k + 3] += v[q][k].w;
                  }
                }
            }
            if (f_ok) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int j = tm * BN + c0 + i;
                if (j < pr.M) ycol[(int64_t)j * pr.ldy] = __float2bfloat16_rn(a[i]);
              }
            }
          }
          if (threadIdx.x == 0) P.counters[gtile] = 0;
        }
        // the flag is rewritten for the next tile only after everyone has read it
        if (!epi_sync()) break;
      }
      u = seg_end;
    }
  }
  __syncthreads();
  if (warp == 5) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, tmem_cols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(P.status, kStatusTimeout);
}

// The same product with data-parallel waves (many token tiles, large activations): each CTA takes
// the whole tiles c, c + G, ... and then its Stream-K share of the tiles of the last, partial wave.
// (A separate kernel: folding the segment loops into the one above measured slower at decode.)
template <bool kF8>
__global__ void __launch_bounds__(threads_of<kF8>(), kF8 ? 1 : 2) k_gemm_tc_waves(const __grid_constant__ Params P) {
  constexpr bool kWaves = true;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const int S = P.stages, BN = P.BN;
  const uint32_t a_atom = BM * BK * 2, b_atom = (uint32_t)BN * BK * 2;
  // k-slices a stage holds: fp8 weights take two, so that each code row of a stage is 128 bytes
  constexpr int KS = kF8 ? 2 : ATOMS;
  const uint32_t a_bytes = KS * a_atom, b_bytes = KS * b_atom;
  // kF8: a stage holds the fp8 codes (a8_bytes: 128 rows x 128 codes) and B; the expanded bf16
  // weights go to a ring of SC slots of a_bytes after the stages
  constexpr uint32_t a8_bytes = BM * BK * KS;
  const uint32_t a_in = kF8 ? a8_bytes : a_bytes;  // bytes of A in a stage
  const uint32_t stage_bytes = a_in + b_bytes;
  const int SC = kF8 ? P.cstages : 0;
  uint8_t *conv = smem + S * stage_bytes;
  uint64_t *full = reinterpret_cast<uint64_t *>(conv + SC * a_bytes);
  uint64_t *empty = full + S;
  uint64_t *cfull = empty + S;    // kF8 [SC]: expanded weights ready (the 128 converter threads)
  uint64_t *cempty = cfull + SC;  // kF8 [SC]: slot read by its MMAs
  uint64_t *accf = cempty + SC;   // [2]
  uint64_t *acce = accf + 2;   // [2]
  uint64_t *drain = acce + 2;
  uint64_t *epi = drain + 1;  // the 128 epilogue threads' own barrier
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(epi + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_last = const_cast<int *>(abort_flag) + 1;
  int *cslot = s_last + 1;  // [kMaxContrib] partial slots of a tile's contributors, in CTA order

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t U = P.total_units, G = gridDim.x;
  const int nseg = kWaves ? P.dp_waves + 1 : 1;
  int sk_b, sk_e;  // the last segment: the Stream-K share (or the split-K range)
  seg_range<kWaves>(P, nseg - 1, sk_b, sk_e);
  if (nseg == 1 && sk_b >= sk_e) return;
  const uint32_t tmem_cols = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int c = 0; c < SC; ++c) {
      tc::mbar_init(&cfull[c], 256);  // both converter groups
      tc::mbar_init(&cempty[c], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], 128);
    }
    tc::mbar_init(drain, 1);
    tc::mbar_init(epi, 128);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 5) tc::tmem_alloc(tmem_slot, tmem_cols);
  if (warp == 4 && lane == 0) {
    for (int p = 0; p < P.nprob; ++p) {
      tc::prefetch_tmap(&P.prob[p].tmA);
      tc::prefetch_tmap(&P.prob[p].tmB);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 4) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_first = tc::policy_evict_first(), pol_normal = tc::policy_evict_normal(),
                     pol_last = tc::policy_evict_last();
      auto pol = [&](int sel) { return sel == 0 ? pol_first : (sel == 1 ? pol_normal : pol_last); };
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int sg = 0; sg < nseg && ok; ++sg) {
      int ub, ue;
      seg_range<kWaves>(P, sg, ub, ue);
      if (ub >= ue) continue;
      // the unit's coordinates, decoded once per segment and then advanced without divisions (this
      // loop paces the copies)
      Unit un = decode_unit(P, ub);
      const Problem *pr = &P.prob[un.p];
      int tm = un.tile % pr->tiles_m, tn = (un.tile / pr->tiles_m) % pr->tiles_n;
      int g = un.tile / (pr->tiles_m * pr->tiles_n);
      // the problem's fields in registers, refreshed when the problem changes
      int kblocks = pr->kblocks, ntiles = pr->tiles, tiles_m = pr->tiles_m, tiles_n = pr->tiles_n, N = pr->N,
          Kg = pr->Kg;
      uint64_t pa = pol(pr->pol_a), pb = pol(pr->pol_b);
      for (int u = ub; u < ue; ++u) {
        if (!(ok = tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag))) break;
        uint8_t *sa = smem + stage * stage_bytes;
        tc::mbar_expect_tx(&full[stage], stage_bytes);
#pragma unroll
        for (int a = 0; a < KS; ++a) {
          const int k0 = (un.kb * KS + a) * BK;
          if (!kF8 || a == 0)  // (fp8: one box of 128 codes a row covers both slices)
            tc::tma_load_2d(sa + a * a_atom, &pr->tmA, &full[stage], k0, g * N + tn * BM, pa);
          tc::tma_load_2d(sa + a_in + a * b_atom, &pr->tmB, &full[stage], g * Kg + k0, tm * BN, pb);
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
        if (++un.kb == kblocks) {  // next tile: token tile fastest, then weight tile, then group
          un.kb = 0;
          if (++un.tile == ntiles) {
            un.tile = 0;
            tm = tn = g = 0;
            if (++un.p < P.nprob) {
              pr = &P.prob[un.p];
              kblocks = pr->kblocks;
              ntiles = pr->tiles;
              tiles_m = pr->tiles_m;
              tiles_n = pr->tiles_n;
              N = pr->N;
              Kg = pr->Kg;
              pa = pol(pr->pol_a);
              pb = pol(pr->pol_b);
            }
          } else if (++tm == tiles_m) {
            tm = 0;
            if (++tn == tiles_n) {
              tn = 0;
              ++g;
            }
          }
        }
      }
      }
      // let every copy this CTA issued land before the CTA can exit
      for (int i = issued - S > 0 ? issued - S : 0; i < issued; ++i) {
        uint64_t *b = &full[i % S];
        const uint32_t par = (uint32_t)((i / S) & 1);
        const uint64_t t0 = tc::global_ns();
        while (!tc::mbar_try_wait(b, par) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int cst = 0;  // kF8: slot of the expanded-weight ring, and its phase
      uint32_t cph = 0;
      int used[2] = {0, 0};
      int buf = 0;
      bool ok = true;
      if (const uint64_t st = stall_ns()) ok = tc::mbar_wait(drain, 0, abort_flag, st);  // test hook
      for (int sg = 0; sg < nseg && ok; ++sg) {
      int ub, ue;
      seg_range<kWaves>(P, sg, ub, ue);
      for (int u = ub; u < ue && ok;) {
        const Unit un = decode_unit(P, u);
        const Problem &pr = P.prob[un.p];
        const int seg_end = min(ue, pr.unit_begin + (un.tile + 1) * pr.kblocks);
        if (!tc::mbar_wait(&acce[buf], (uint32_t)(used[buf] & 1) ^ 1u, abort_flag)) break;
        tc::tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * BN);
        bool first = true;
        for (; u < seg_end; ++u) {
          if (!tc::mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          if constexpr (kF8) {  // the expanded weights of this unit
            if (!tc::mbar_wait(&cfull[cst], cph, abort_flag)) {
              ok = false;
              break;
            }
          }
          tc::tc_fence_after();
          const uint32_t sa = tc::smem_u32(smem + stage * stage_bytes);
          const uint32_t sa_w = kF8 ? tc::smem_u32(conv + cst * a_bytes) : sa;
#pragma unroll
          for (int a = 0; a < KS; ++a) {
            const uint64_t ad = tc::sdesc_sw128(sa_w + a * a_atom, 16, 1024);
            const uint64_t bd = tc::sdesc_sw128(sa + a_in + a * b_atom, 16, 1024);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              tc::mma_bf16(d, ad + 2ull * k, bd + 2ull * k, idesc, (first && a == 0 && k == 0) ? 0u : 1u);
          }
          first = false;
          tc::mma_commit(&empty[stage]);
          if constexpr (kF8) {
            tc::mma_commit(&cempty[cst]);
            if (++cst == SC) {
              cst = 0;
              cph ^= 1u;
            }
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit(&accf[buf]);
        ++used[buf];
        buf ^= 1;
      }
      }
      // every MMA issued has completed once this arrives
      tc::mma_commit(drain);
      const uint64_t t0 = tc::global_ns();
      while (!tc::mbar_try_wait(drain, 0) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
      }
    }
  } else if (kF8 && warp >= 6) {
    // ---------------------------------------------------------------- fp8 expansion (warps 6-9)
    // the second half of every stage's codes, in unit order, beside the epilogue warps' first half
    const int t = threadIdx.x - 192;
    int rst = 0, cst = 0;
    uint32_t rph = 0, cph = 0;
    for (int sg = 0; sg < nseg; ++sg) {
      int ub, ue;
      seg_range<kWaves>(P, sg, ub, ue);
      bool okc = true;
      for (int v = ub; v < ue; ++v) {
        const Unit un = decode_unit(P, v);
        const Problem &pr = P.prob[un.p];
        const int rest = un.tile / pr.tiles_m, tn = rest % pr.tiles_n, g = rest / pr.tiles_n;
        const int row0 = g * pr.N + tn * BM, kcol = un.kb;
        const float sc0 = fp8_stage_scale(pr.scale, pr.ld_scale, row0, pr.N * pr.groups, kcol);
        if (!(okc = tc::mbar_wait(&full[rst], rph, abort_flag))) break;
        if (!(okc = tc::mbar_wait(&cempty[cst], cph ^ 1u, abort_flag))) break;
        fp8_expand_half<4>(smem + rst * stage_bytes, conv + cst * a_bytes, pr.scale, pr.ld_scale, row0,
                           pr.N * pr.groups, kcol, t, sc0);
        fence_proxy_async_smem();
        tc::mbar_arrive(&cfull[cst]);
        if (++rst == S) {
          rst = 0;
          rph ^= 1u;
        }
        if (++cst == SC) {
          cst = 0;
          cph ^= 1u;
        }
      }
      if (!okc) break;
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- epilogue (warps 0-3)
    const int row = warp * 32 + lane;  // feature within the tile
    int done[2] = {0, 0};
    uint32_t epi_uses = 0;
    auto epi_sync = [&]() -> bool {
      tc::mbar_arrive(epi);
      return tc::mbar_wait(epi, (epi_uses++) & 1u, abort_flag);
    };
    // kF8: expand the weights of units [v0, v1) of one tile (first k-slice kb0, weight rows from
    // row0), in unit order, into the expanded-weight ring
    int rst = 0, cst = 0;
    uint32_t rph = 0, cph = 0;
    auto convert_units = [&](int v0, int v1, const Problem &pr, int row0, int kb0) -> bool {
      for (int v = v0; v < v1; ++v) {
        const int kcol = kb0 + v - v0;  // (a unit is one 128-wide scale column)
        const float sc0 = fp8_stage_scale(pr.scale, pr.ld_scale, row0, pr.N * pr.groups, kcol);
        if (!tc::mbar_wait(&full[rst], rph, abort_flag)) return false;
        if (!tc::mbar_wait(&cempty[cst], cph ^ 1u, abort_flag)) return false;
        fp8_expand_half<0>(smem + rst * stage_bytes, conv + cst * a_bytes, pr.scale, pr.ld_scale, row0,
                           pr.N * pr.groups, kcol, threadIdx.x, sc0);
        fence_proxy_async_smem();
        tc::mbar_arrive(&cfull[cst]);
        if (++rst == S) {
          rst = 0;
          rph ^= 1u;
        }
        if (++cst == SC) {
          cst = 0;
          cph ^= 1u;
        }
      }
      return true;
    };
    int buf = 0;
    // the Stream-K share's first tile (its partial goes to slot 0, the last tile's to slot 1)
    const int first_tile_global = [&] {
      if (sk_b >= sk_e) return -1;
      const Unit f = decode_unit(P, sk_b);
      return P.prob[f.p].tile_begin + f.tile;
    }();
    const int sk0 = kWaves ? P.sk_unit0 : 0;
    const int64_t Usk = U - sk0;
    bool eok = true;
    for (int sg = 0; sg < nseg && eok; ++sg) {
    int ub, ue;
    seg_range<kWaves>(P, sg, ub, ue);
    for (int u = ub; u < ue;) {
      const Unit un = decode_unit(P, u);
      const Problem &pr = P.prob[un.p];
      const int tile_u0 = pr.unit_begin + un.tile * pr.kblocks, tile_u1 = tile_u0 + pr.kblocks;
      const int seg_end = min(ue, tile_u1);
      const bool whole = (u == tile_u0) && (seg_end == tile_u1);
      const int tm = un.tile % pr.tiles_m, rest = un.tile / pr.tiles_m;
      const int tn = rest % pr.tiles_n, g = rest / pr.tiles_n;
      const int f = tn * BM + row;
      const bool f_ok = f < pr.N;
      bf16 *ycol = pr.y + (int64_t)g * pr.N + f;
      const int gtile = pr.tile_begin + un.tile;
      if constexpr (kF8) {
        if (!(eok = convert_units(u, seg_end, pr, g * pr.N + tn * BM, un.kb))) break;
      }
      if (!(eok = tc::mbar_wait(&accf[buf], (uint32_t)(done[buf] & 1), abort_flag))) break;
      tc::tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * BN);
      if (P.split_S > 0) {
        // split-K: this CTA's partial sum for (tile, k-range) as f32, coalesced over features
        const int sp = blockIdx.x % P.split_S;
        float *pcol = pr.part + (int64_t)g * pr.N + f;
        for (int c0 = 0; c0 < BN; c0 += 16) {
          uint32_t r[16];
          tc::tmem_ld16(taddr + (uint32_t)c0, r);
          tc::tmem_ld_wait();
          if (f_ok) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j = tm * BN + c0 + i;
              if (j < pr.M) pcol[((int64_t)sp * pr.M + j) * pr.ldp] = __uint_as_float(r[i]);
            }
          }
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&acce[buf]);
        ++done[buf];
        buf ^= 1;
        u = seg_end;
        continue;
      }
      const int slot = (int)blockIdx.x * 2 + (gtile == first_tile_global ? 0 : 1);
      // partial tile layout: 4-column groups, the group's 128 rows contiguous (row r, columns 4c..4c+3
      // at (c * BM + r) * 4), so that a warp's 16-byte stores and loads cover 512 contiguous bytes
      float *mine = P.partials + (size_t)slot * BM * BN;
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t r[16];
        tc::tmem_ld16(taddr + (uint32_t)c0, r);
        tc::tmem_ld_wait();
        if (whole) {
          if (f_ok) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j = tm * BN + c0 + i;
              if (j < pr.M) ycol[(int64_t)j * pr.ldy] = __float2bfloat16_rn(__uint_as_float(r[i]));
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4 *>(mine + ((size_t)((c0 + i) >> 2) * BM + row) * 4) =
                make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]), __uint_as_float(r[i + 2]),
                            __uint_as_float(r[i + 3]));
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&acce[buf]);
      ++done[buf];
      buf ^= 1;
      if (!whole) {
        // Stream-K fixup: the last contributor of this tile sums the partials in CTA order (published
        // and acquired as in the kernel above).
        if (!(eok = epi_sync())) break;
        const int64_t c_first = unit_owner(tile_u0 - sk0, Usk, G), c_last = unit_owner(tile_u1 - 1 - sk0, Usk, G);
        if (threadIdx.x == 0) {
          const int old = atom_add_acq_rel_gpu(&P.counters[gtile], 1);
          *s_last = (old == (int)(c_last - c_first)) ? 1 : 0;
        }
        if (!(eok = epi_sync())) break;
        if (*s_last) {
          const int nc = (int)(c_last - c_first + 1);
          for (int i = threadIdx.x; i < nc; i += 128) {
            const int64_t c = c_first + i;
            const Unit f0 = decode_unit(P, sk0 + (int)cta_start(c, Usk, G));
            cslot[i] = (int)c * 2 + (gtile == P.prob[f0.p].tile_begin + f0.tile ? 0 : 1);
          }
          if (!(eok = epi_sync())) break;
          // sum the contributors' rows in CTA order, four contributors' 16-column chunks in flight
          const float *base = P.partials + (size_t)row * 4;
          for (int c0 = 0; c0 < BN; c0 += 16) {
            float a[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) a[i] = 0.f;
            for (int i = 0; i < nc; i += 4) {
              float4 v[4][4];
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (i + q < nc) {
                  const float *src = base + (size_t)cslot[i + q] * BM * BN + (size_t)(c0 >> 2) * BM * 4;
#pragma unroll
                  for (int k = 0; k < 4; ++k) v[q][k] = __ldcg(reinterpret_cast<const float4 *>(src + (size_t)k * BM * 4));
                }
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (i + q < nc) {
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    a[4 * k] += v[q][k].x;
                    a[4 * k + 1] += v[q][k].y;
                    a[4 * k + 2] += v[q][k].z;
                    a[4 * k + 3] += v[q][k].w;
                  }
                }
            }
            if (f_ok) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int j = tm * BN + c0 + i;
                if (j < pr.M) ycol[(int64_t)j * pr.ldy] = __float2bfloat16_rn(a[i]);
              }
            }
          }
          if (threadIdx.x == 0) P.counters[gtile] = 0;
        }
        // the flag is rewritten for the next tile only after everyone has read it
        if (!(eok = epi_sync())) break;
      }
      u = seg_end;
    }
    }
  }
  __syncthreads();
  if (warp == 5) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, tmem_cols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(P.status, kStatusTimeout);
}

// ---- pairs: clusters of two CTAs sharing the token tile ----------------------------------------------
// For launches with many token tiles: the two CTAs of a cluster take the weight tiles 2j and 2j + 1 of
// one 256-token tile; each copies half of the activation tile (128 tokens) and multicasts it into both
// CTAs' stages, so that a CTA reads 32 instead of 48 KiB from L2 per 64-wide k-slice (the prefill
// projections are bound by that traffic).  Whole pair tiles in waves (cluster v takes pair tiles v,
// v + NP, ...; token tile fastest, so the clusters in flight share the weight tiles too), no Stream-K.
// A stage is refilled only once both CTAs' MMAs have read it: its empty barrier counts the commits of
// both, each MMA issuer committing to the two CTAs' barriers at once.
__device__ __forceinline__ void tma_load_2d_mc(void *dst, const CUtensorMap *tm, uint64_t *bar, int c0, int c1,
                                               uint16_t mask, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5, %6;" ::"r"(tc::smem_u32(dst)),
      "l"((uint64_t)tm), "r"(tc::smem_u32(bar)), "r"(c0), "r"(c1), "h"(mask), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void mma_commit_mc(uint64_t *bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   tc::smem_u32(bar)),
               "h"(mask)
               : "memory");
}

// Pair tile pt of the launch: problem, token tile, weight-tile pair, group.  A problem with an odd
// number of weight tiles has a last pair whose second tile lies past N (its copies read zeros or the
// next group's rows, its stores are masked).
struct PairTile {
  int p, tm, j, g;
};
__device__ __forceinline__ int pair_tiles_of(const Problem &pr) { return pr.tiles_m * ((pr.tiles_n + 1) / 2) * pr.groups; }
__device__ __forceinline__ PairTile decode_pair(const Params &P, int pt) {
  int p = 0, begin = 0;
  while (p + 1 < P.nprob && pt >= begin + pair_tiles_of(P.prob[p])) begin += pair_tiles_of(P.prob[p++]);
  const Problem &pr = P.prob[p];
  const int local = pt - begin, half_n = (pr.tiles_n + 1) / 2;
  return PairTile{p, local % pr.tiles_m, (local / pr.tiles_m) % half_n, local / (pr.tiles_m * half_n)};
}

constexpr int kPairBN = 256;  // tokens of a tile (the pair's shared operand)

__global__ void __launch_bounds__(kThreads, 1) k_gemm_tc_pairs(const __grid_constant__ Params P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const int S = P.stages;
  constexpr uint32_t a_bytes = BM * BK * 2, b_half = 128 * BK * 2, b_bytes = 2 * b_half;
  constexpr uint32_t stage_bytes = a_bytes + b_bytes;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S * stage_bytes);
  uint64_t *empty = full + S;
  uint64_t *accf = empty + S;  // [2]
  uint64_t *acce = accf + 2;   // [2]
  uint64_t *drain = acce + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)tc::cluster_ctarank();
  const int v0 = blockIdx.x >> 1, NP = gridDim.x >> 1;
  const int KSP = P.ksplit > 1 ? P.ksplit : 1;
  const int W = P.pt_count * KSP;  // work items: (pair tile, k-range)
  // work item w: its pair tile and k-slices [kb0, kb1)
  auto item = [&](int w, int &pt, int &kb0, int &kb1, int kbl) {
    pt = P.pt_begin + w / KSP;
    const int sp = w % KSP;
    kb0 = sp * kbl / KSP;
    kb1 = (sp + 1) * kbl / KSP;
  };
  constexpr uint16_t kBoth = 3;
  constexpr uint32_t tmem_cols = 2 * kPairBN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 2);  // both CTAs' MMA commits
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], 128);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 5) tc::tmem_alloc(tmem_slot, tmem_cols);
  if (warp == 4 && lane == 0) {
    for (int p = 0; p < P.nprob; ++p) {
      tc::prefetch_tmap(&P.prob[p].tmA);
      tc::prefetch_tmap(&P.prob[p].tmB);
    }
  }
  tc::tc_fence_before();
  // the peer's barriers are initialised before any copy or commit of this CTA reaches them
  tc::cluster_sync();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 4) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_normal = tc::policy_evict_normal(), pol_last = tc::policy_evict_last();
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int w = v0; w < W && ok; w += NP) {
        int pt, kb0, kb1;
        item(w, pt, kb0, kb1, P.prob[0].kblocks);
        const PairTile q = decode_pair(P, pt);
        const Problem &pr = P.prob[q.p];
        if (KSP == 1) kb1 = pr.kblocks;
        const int tn = 2 * q.j + rank;
        const uint64_t pa = pr.pol_a == 2 ? pol_last : pol_normal, pb = pr.pol_b == 2 ? pol_last : pol_normal;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!(ok = tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag))) break;
          uint8_t *sa = smem + stage * stage_bytes;
          tc::mbar_expect_tx(&full[stage], stage_bytes);
          const int k0 = kb * BK;
          tc::tma_load_2d(sa, &pr.tmA, &full[stage], k0, q.g * pr.N + tn * BM, pa);
          tma_load_2d_mc(sa + a_bytes + rank * b_half, &pr.tmB, &full[stage], q.g * pr.Kg + k0,
                         q.tm * kPairBN + rank * 128, kBoth, pb);
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // every copy into this CTA has landed before it can exit (the peer's halves included)
      for (int i = issued - S > 0 ? issued - S : 0; i < issued; ++i) {
        const uint64_t t0 = tc::global_ns();
        while (!tc::mbar_try_wait(&full[i % S], (uint32_t)((i / S) & 1)) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(BM, kPairBN);
      int stage = 0, buf = 0;
      uint32_t phase = 0;
      int used[2] = {0, 0};
      bool ok = true;
      for (int w = v0; w < W && ok; w += NP) {
        int pt, kb0, kb1;
        item(w, pt, kb0, kb1, P.prob[0].kblocks);
        const PairTile q = decode_pair(P, pt);
        if (KSP == 1) kb1 = P.prob[q.p].kblocks;
        if (!(ok = tc::mbar_wait(&acce[buf], (uint32_t)(used[buf] & 1) ^ 1u, abort_flag))) break;
        tc::tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * kPairBN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!(ok = tc::mbar_wait(&full[stage], phase, abort_flag))) break;
          tc::tc_fence_after();
          const uint32_t sa = tc::smem_u32(smem + stage * stage_bytes);
          const uint64_t ad = tc::sdesc_sw128(sa, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(sa + a_bytes, 16, 1024);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc::mma_bf16(d, ad + 2ull * k, bd + 2ull * k, idesc, (kb == kb0 && k == 0) ? 0u : 1u);
          mma_commit_mc(&empty[stage], kBoth);  // both CTAs may refill their halves of this stage
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit(&accf[buf]);
        ++used[buf];
        buf ^= 1;
      }
      // every MMA issued (and every commit it makes to either CTA) has completed once this arrives
      tc::mma_commit(drain);
      const uint64_t t0 = tc::global_ns();
      while (!tc::mbar_try_wait(drain, 0) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
      }
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- epilogue (warps 0-3)
    const int row = warp * 32 + lane;  // feature within the tile
    int buf = 0, done[2] = {0, 0};
    for (int w = v0; w < W; w += NP) {
      int pt, kb0, kb1;
      item(w, pt, kb0, kb1, P.prob[0].kblocks);
      const PairTile q = decode_pair(P, pt);
      const Problem &pr = P.prob[q.p];
      const int f = (2 * q.j + rank) * BM + row;
      const bool f_ok = f < pr.N;
      bf16 *ycol = pr.y ? pr.y + (int64_t)q.g * pr.N + f : nullptr;
      float *pcol = pr.part ? pr.part + (int64_t)q.g * pr.N + f : nullptr;  // f32 result (one split slice)
      // a k-range's partial sums: [split][item][token in tile][feature in pair], lanes on features
      float *tcol = KSP > 1 ? P.tail_part + ((size_t)((w % KSP) * P.pt_count + (pt - P.pt_begin)) * kPairBN) * 256 +
                                  rank * BM + row
                            : nullptr;
      if (!tc::mbar_wait(&accf[buf], (uint32_t)(done[buf] & 1), abort_flag)) break;
      tc::tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * kPairBN);
      for (int c0 = 0; c0 < kPairBN; c0 += 16) {
        uint32_t r[16];
        tc::tmem_ld16(taddr + (uint32_t)c0, r);
        tc::tmem_ld_wait();
        if (tcol) {
#pragma unroll
          for (int i = 0; i < 16; ++i) tcol[(size_t)(c0 + i) * 256] = __uint_as_float(r[i]);
        } else if (f_ok && pcol) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int jt = q.tm * kPairBN + c0 + i;
            if (jt < pr.M) pcol[(int64_t)jt * pr.ldp] = __uint_as_float(r[i]);
          }
        } else if (f_ok) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int jt = q.tm * kPairBN + c0 + i;
            if (jt < pr.M) ycol[(int64_t)jt * pr.ldy] = __float2bfloat16_rn(__uint_as_float(r[i]));
          }
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&acce[buf]);
      ++done[buf];
      buf ^= 1;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  // neither CTA exits while the other may still copy into it or commit to its barriers
  tc::cluster_sync();
  if (warp == 5) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, tmem_cols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(P.status, kStatusTimeout);
}

// The split tail's sums: block (item, token) adds the k-ranges' partials of one token row of a pair
// tile (256 features, a thread each) and writes them as bf16.
__global__ void __launch_bounds__(256) k_pair_tail_sum(const float *__restrict__ part, int ksplit, int pt_begin,
                                                       int pt_count, int tiles_m, int half_n, int M, int N,
                                                       bf16 *__restrict__ y, int ldy) {
  const int w = blockIdx.x / kPairBN, tok = blockIdx.x % kPairBN, f = threadIdx.x;
  const int pt = pt_begin + w;
  const int tm = pt % tiles_m, j = (pt / tiles_m) % half_n;
  const int row = tm * kPairBN + tok, col = j * 2 * BM + f;
  float acc = 0.f;
  for (int sp = 0; sp < ksplit; ++sp) acc += __ldcg(part + ((size_t)(sp * pt_count + w) * kPairBN + tok) * 256 + f);
  if (row < M && col < N) y[(int64_t)row * ldy + col] = __float2bfloat16_rn(acc);
}

// ---- host ---------------------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once per process (a function-local static: initialised once even with several threads).
EncodeTiledFn encoder() {
  static const EncodeTiledFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

// 2-D bf16 map of a row-major [outer][inner] array with row stride `ld` elements, 128B swizzle.
bool map_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
            uint32_t box_outer) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  if (((uintptr_t)base & 15) || (ld * 2) % 16) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D uint8 map (fp8 weight codes) of a row-major [outer][inner] byte array with row stride `ld`
// bytes, unswizzled.
bool map_2d_u8(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
               uint32_t box_outer) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  if (((uintptr_t)base & 15) || ld % 16) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gemm

bool tma_map_2d_bf16(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
                     uint32_t box_outer) {
  return gemm::map_2d(m, base, inner, outer, ld, box_inner, box_outer);
}

// L2 policies: a weight read by one token tile only (few tokens) streams past evict-first; one
// re-read by several token tiles stays normal.  Activations that all weight tiles re-read stay
// evict-last while they are small next to L2, normal otherwise.
static void set_policies(gemm::Problem &p, const LinearProblem &q, int M) {
  p.pol_a = p.tiles_m == 1 ? 0 : 1;
  const size_t x_bytes = (size_t)M * q.K * q.groups * 2;
  p.pol_b = x_bytes <= ((size_t)16 << 20) ? 2 : 1;
}
// The kernels take the launch's policies from its first problem: problems that disagree get normal.
static void unify_policies(gemm::Params &P, int nprob) {
  for (int i = 1; i < nprob; ++i) {
    if (P.prob[i].pol_a != P.prob[0].pol_a) P.prob[0].pol_a = 1;
    if (P.prob[i].pol_b != P.prob[0].pol_b) P.prob[0].pol_b = 1;
  }
  for (int i = 1; i < nprob; ++i) {
    P.prob[i].pol_a = P.prob[0].pol_a;
    P.prob[i].pol_b = P.prob[0].pol_b;
  }
}

int gemm_tc_bn(int M, bool f8) {
  if (M > 256) return f8 ? 128 : 256;  // (fp8 stages hold two k-slices: 256-token tiles leave room for one)
  int bn = (M + 15) / 16 * 16;
  return bn < 16 ? 16 : bn;
}

// Launch up to kMaxProblems products that share M (token count) in one persistent Stream-K grid.
cudaError_t launch_gemm_tc(const LinearProblem *probs, int nprob, float *ws, size_t ws_bytes, int num_sms,
                           int *status, cudaStream_t s, int *kernels) {
  using namespace gemm;
  if (nprob <= 0 || nprob > kMaxProblems) return cudaErrorInvalidValue;
  const int M = probs[0].M;
  Params P;
  memset(&P, 0, sizeof(P));
  // fp8 weights: every problem of the launch; a stage holds two k-slices of codes (128 bytes a
  // weight row, one TMA box) and of activations, and a ring of two expanded bf16 stages feeds the MMA
  const bool f8 = probs[0].W8 != nullptr;
  for (int i = 1; i < nprob; ++i)
    if ((probs[i].W8 != nullptr) != f8) return cudaErrorInvalidValue;
  P.BN = gemm_tc_bn(M, f8);
  const int ks = f8 ? 2 : ATOMS;  // k-slices a stage (fp8: two, so each code row is 128 bytes)
  const int stage_bytes = f8 ? 2 * (BM * BK + P.BN * BK * 2) : ATOMS * (BM * BK * 2 + P.BN * BK * 2);
  // one CTA per SM: two per SM (five stages each) measured slower at decode, because twice the CTAs
  // split each tile's k-range twice as often and the Stream-K fixups dominate
  const int per_sm = 1;
  P.cstages = f8 ? 2 : 0;
  const int conv_bytes = P.cstages * 2 * BM * BK * 2;
  // (fp8: the shared memory left beside the expansion ring, short of the barriers and the 1 KB alignment)
  P.stages = per_sm == 2 ? std::min(5, (100 * 1024) / stage_bytes)
                         : std::min(8, ((f8 ? 222 : 200) * 1024 - conv_bytes) / stage_bytes);
  if (P.stages < 2) return cudaErrorInvalidValue;
  // many token tiles (prefill): clusters of two CTAs on adjacent weight tiles sharing the token tile
  const bool pairs = !f8 && P.BN == 256 && ATOMS == 1 && M >= 2048;
  for (int i = 0; i < nprob; ++i)  // an f32 result (a split-K slice layout) only from the paired kernel
    if (probs[i].part && !pairs) return cudaErrorInvalidValue;
  int units = 0, tiles = 0;
  for (int i = 0; i < nprob; ++i) {
    const LinearProblem &q = probs[i];
    if (q.M != M) return cudaErrorInvalidValue;
    Problem &p = P.prob[i];
    if (f8) {
      if (!q.w8_scale || !map_2d_u8(&p.tmA, q.W8, (uint64_t)q.K, (uint64_t)q.N * q.groups, (uint64_t)q.ldw, 2 * BK, BM))
        return cudaErrorInvalidValue;
      p.scale = q.w8_scale;
      p.ld_scale = (q.K + 127) / 128;
    } else if (!map_2d(&p.tmA, q.W, (uint64_t)q.K, (uint64_t)q.N * q.groups, (uint64_t)q.ldw, BK, BM)) {
      return cudaErrorInvalidValue;
    }
    if (!map_2d(&p.tmB, q.x, (uint64_t)q.K * q.groups, (uint64_t)M, (uint64_t)q.ldx, BK,
                (uint32_t)(pairs ? P.BN / 2 : P.BN)))  // pairs: each CTA copies half the token tile
      return cudaErrorInvalidValue;
    p.y = q.y;
    p.ldy = q.ldy;
    p.part = q.part;
    p.ldp = q.ldp;
    p.N = q.N;
    p.M = M;
    p.groups = q.groups;
    p.Kg = q.K;
    p.kblocks = (q.K + BK * ks - 1) / (BK * ks);
    p.tiles_n = (q.N + BM - 1) / BM;
    p.tiles_m = (M + P.BN - 1) / P.BN;
    p.tiles = p.tiles_n * p.tiles_m * q.groups;
    set_policies(p, q, M);
    p.unit_begin = units;
    p.tile_begin = tiles;
    units += p.tiles * p.kblocks;
    tiles += p.tiles;
  }
  P.nprob = nprob;
  for (int q = 0; q < nprob; ++q) P.early_dependents |= probs[q].early_dependents;
  for (int q = 0; q < nprob; ++q) P.pdl |= probs[q].pdl;
  unify_policies(P, nprob);
  P.total_units = units;
  P.total_tiles = tiles;
  P.split_S = 0;
  if (tiles > kCounterInts) return cudaErrorInvalidValue;
  const size_t part_per_cta = (size_t)2 * BM * P.BN * sizeof(float);
  if (ws_bytes < kCounterBytes + part_per_cta) return cudaErrorInvalidValue;
  const int ws_grid = (int)std::min<size_t>((ws_bytes - kCounterBytes) / part_per_cta, (size_t)(kMaxContrib - 1));
  int grid = std::min(std::min(per_sm * num_sms, units), ws_grid);
  {
    // weight streaming (one token tile): a slightly smaller grid whose Stream-K ranges are whole
    // tiles needs no fixup at all -- take it when one exists within 80% of the SMs (the problems of
    // the launch sharing one k-slice count).  Compute-bound launches keep every SM.
    bool same_kb = P.prob[0].tiles_m == 1;
    for (int i = 1; i < nprob; ++i) same_kb = same_kb && P.prob[i].kblocks == P.prob[0].kblocks;
    const int kb = P.prob[0].kblocks;
    int pick = 0;
    for (int gsz = grid; same_kb && gsz * 5 >= grid * 4 && !pick; --gsz)
      if (units % gsz == 0 && (units / gsz) % kb == 0) pick = gsz;
    // else one whose ranges are equal fractions of a tile: every fixup then has the same few
    // contributors, all finishing together
    for (int gsz = grid; same_kb && gsz * 5 >= grid * 4 && !pick; --gsz)
      if (units % gsz == 0 && kb % (units / gsz) == 0) pick = gsz;
    if (pick) grid = pick;
  }
  // many token tiles and large activations (prefill): whole tiles in data-parallel waves first, so that the tiles in
  // flight at a time are consecutive ones whose operands fit in L2 together (contiguous Stream-K
  // ranges would have every CTA stream its own far-apart tiles, re-reading each operand tile from
  // DRAM); Stream-K only over the tiles of the last, partial wave.  Few token tiles: Stream-K alone.
  bool many_m = true;  // many token tiles, and activations well beyond what L2 holds
  for (int i = 0; i < nprob; ++i)
    many_m = many_m && P.prob[i].tiles_m > 1 && (size_t)M * probs[i].K * probs[i].groups * 2 > kWaveActBytes;
  P.dp_waves = many_m ? tiles / grid : 0;
  {
    // the Stream-K part must give every CTA at least one unit (the fixup counts every CTA between a
    // tile's first and last owner as a contributor): keep one more wave in it when it would not
    auto unit_of_tile = [&](int t) {
      int p = 0;
      while (p + 1 < nprob && t >= P.prob[p + 1].tile_begin) ++p;
      return t >= tiles ? units : P.prob[p].unit_begin + (t - P.prob[p].tile_begin) * P.prob[p].kblocks;
    };
    if (P.dp_waves > 0 && units - unit_of_tile(P.dp_waves * grid) < grid && units - unit_of_tile(P.dp_waves * grid) > 0)
      --P.dp_waves;
  }
  {
    const int t = P.dp_waves * grid;  // first tile of the Stream-K part
    int p = 0;
    while (p + 1 < nprob && t >= P.prob[p + 1].tile_begin) ++p;
    P.sk_unit0 = t >= tiles ? units : P.prob[p].unit_begin + (t - P.prob[p].tile_begin) * P.prob[p].kblocks;
  }
  P.counters = reinterpret_cast<int *>(ws);
  P.partials = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ws) + kCounterBytes);
  P.status = status;
  if (pairs || P.dp_waves > 0) P.pdl = 0;  // (the programmatic prologue is k_gemm_tc's)
  if (pairs) {
    const size_t psmem = 1024 + (size_t)P.stages * stage_bytes + (size_t)(2 * P.stages + 5) * 8 + 16;
    static SmemAttr attr_pairs;
    cudaError_t e = attr_pairs.ensure((const void *)k_gemm_tc_pairs, 227 * 1024);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = psmem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    // as many clusters as fit on the GPU at once (an SM each CTA), at most one per pair tile
    cfg.gridDim = dim3(2 * (num_sms / 2));
    int nclusters = 0;
    e = cudaOccupancyMaxActiveClusters(&nclusters, (const void *)k_gemm_tc_pairs, &cfg);
    if (e != cudaSuccess) return e;
    int pair_tiles = 0;
    for (int i = 0; i < nprob; ++i)
      pair_tiles += P.prob[i].tiles_m * ((P.prob[i].tiles_n + 1) / 2) * P.prob[i].groups;
    nclusters = std::min(std::max(nclusters, 1), std::max(1, pair_tiles));
    cfg.gridDim = dim3(2 * nclusters);
    P.pt_begin = 0;
    P.pt_count = pair_tiles;
    P.ksplit = 1;
    P.tail_part = nullptr;
    // the last, partial wave of whole pair tiles split by k-range over the clusters (one problem with
    // a bf16 result): the k-ranges' f32 sums go to the workspace, and a small kernel adds them
    const int full = (pair_tiles / nclusters) * nclusters, tail = pair_tiles - full;
    int ks = 0;
    if (kernels && tail > 0 && full > 0 && nprob == 1 && !probs[0].part && probs[0].groups == 1) {
      const int kbl = P.prob[0].kblocks;
      for (int c = 2; c <= 8; ++c)
        if (tail * c <= nclusters && kbl % c == 0 && kbl / c >= 4) ks = c;
      if (ks && ws_bytes < kCounterBytes + (size_t)ks * tail * kPairBN * 256 * sizeof(float)) ks = 0;
    }
    if (ks) P.pt_count = full;
    e = cudaLaunchKernelEx(&cfg, k_gemm_tc_pairs, P);
    if (e != cudaSuccess) return e;
    if (kernels) *kernels = 1;
    if (!ks) return cudaGetLastError();
    Params P2 = P;
    P2.pt_begin = full;
    P2.pt_count = tail;
    P2.ksplit = ks;
    P2.tail_part = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ws) + kCounterBytes);
    cfg.gridDim = dim3(2 * tail * ks);
    e = cudaLaunchKernelEx(&cfg, k_gemm_tc_pairs, P2);
    if (e != cudaSuccess) return e;
    const Problem &q0 = P.prob[0];
    k_pair_tail_sum<<<tail * kPairBN, 256, 0, s>>>(P2.tail_part, ks, full, tail, q0.tiles_m, (q0.tiles_n + 1) / 2, M,
                                                   q0.N, q0.y, q0.ldy);
    *kernels = 3;
    return cudaGetLastError();
  }
  const size_t smem = 1024 + (size_t)P.stages * stage_bytes + conv_bytes +
                      (size_t)(2 * P.stages + 2 * P.cstages + 8) * 8 + 64 + kMaxContrib * sizeof(int);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  static SmemAttr attr, attr_waves, attr8, attr8_waves;
  const void *fn = P.dp_waves > 0 ? (f8 ? (const void *)k_gemm_tc_waves<true> : (const void *)k_gemm_tc_waves<false>)
                                  : (f8 ? (const void *)k_gemm_tc<true> : (const void *)k_gemm_tc<false>);
  {
    SmemAttr &at = P.dp_waves > 0 ? (f8 ? attr8_waves : attr_waves) : (f8 ? attr8 : attr);
    cudaError_t e = at.ensure(fn, 227 * 1024);
    if (e != cudaSuccess) return e;
  }
  if (P.dp_waves > 0) {
    if (f8)
      k_gemm_tc_waves<true><<<grid, kThreadsF8, smem, s>>>(P);
    else
      k_gemm_tc_waves<false><<<grid, kThreads, smem, s>>>(P);
  } else if (P.pdl) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(f8 ? kThreadsF8 : kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    const cudaError_t e = f8 ? cudaLaunchKernelEx(&cfg, k_gemm_tc<true>, P) : cudaLaunchKernelEx(&cfg, k_gemm_tc<false>, P);
    if (e != cudaSuccess) return e;
  } else {
    if (f8)
      k_gemm_tc<true><<<grid, kThreadsF8, smem, s>>>(P);
    else
      k_gemm_tc<false><<<grid, kThreads, smem, s>>>(P);
  }
  return cudaGetLastError();
}

int gemm_tc_split_count(const LinearProblem *probs, int nprob, int max_ctas, int max_S) {
  using namespace gemm;
  const int BN = gemm_tc_bn(probs[0].M, false);
  int tiles = 0;
  for (int i = 0; i < nprob; ++i)
    tiles += ((probs[i].N + BM - 1) / BM) * ((probs[i].M + BN - 1) / BN) * probs[i].groups;
  const int kblocks = (probs[0].K + BK * ATOMS - 1) / (BK * ATOMS);
  int best = 1;
  for (int s = 1; s <= kblocks && s <= max_S; ++s)
    if (kblocks % s == 0 && (int64_t)tiles * s <= max_ctas) best = s;
  return best;
}

cudaError_t launch_gemm_tc_split(const LinearProblem *probs, int nprob, int S, int *status, cudaStream_t s) {
  using namespace gemm;
  if (nprob <= 0 || nprob > kMaxProblems || S <= 0) return cudaErrorInvalidValue;
  const int M = probs[0].M, K = probs[0].K;
  Params P;
  memset(&P, 0, sizeof(P));
  P.BN = gemm_tc_bn(M, false);
  const int stage_bytes = ATOMS * (BM * BK * 2 + P.BN * BK * 2);
  P.stages = std::min(8, (200 * 1024) / stage_bytes);
  if (P.stages < 2) return cudaErrorInvalidValue;
  int units = 0, tiles = 0;
  for (int i = 0; i < nprob; ++i) {
    const LinearProblem &q = probs[i];
    if (q.M != M || q.K != K || !q.part || q.W8) return cudaErrorInvalidValue;
    Problem &p = P.prob[i];
    if (!map_2d(&p.tmA, q.W, (uint64_t)q.K, (uint64_t)q.N * q.groups, (uint64_t)q.ldw, BK, BM)) return cudaErrorInvalidValue;
    if (!map_2d(&p.tmB, q.x, (uint64_t)q.K * q.groups, (uint64_t)M, (uint64_t)q.ldx, BK, (uint32_t)P.BN))
      return cudaErrorInvalidValue;
    p.y = q.y;
    p.part = q.part;
    p.ldp = q.ldp;
    p.ldy = q.ldy;
    p.N = q.N;
    p.M = M;
    p.groups = q.groups;
    p.Kg = q.K;
    p.kblocks = (q.K + BK * ATOMS - 1) / (BK * ATOMS);
    if (p.kblocks % S) return cudaErrorInvalidValue;
    p.tiles_n = (q.N + BM - 1) / BM;
    p.tiles_m = (M + P.BN - 1) / P.BN;
    p.tiles = p.tiles_n * p.tiles_m * q.groups;
    set_policies(p, q, M);
    p.unit_begin = units;
    p.tile_begin = tiles;
    units += p.tiles * p.kblocks;
    tiles += p.tiles;
  }
  P.nprob = nprob;
  for (int q = 0; q < nprob; ++q) P.early_dependents |= probs[q].early_dependents;
  unify_policies(P, nprob);
  P.total_units = units;
  P.total_tiles = tiles;
  P.split_S = S;
  P.dp_waves = 0;
  P.sk_unit0 = 0;
  P.status = status;
  const size_t smem = 1024 + (size_t)P.stages * stage_bytes + 256 + kMaxContrib * sizeof(int);
  static SmemAttr attr;
  {
    cudaError_t e = attr.ensure((const void *)k_gemm_tc<false>, 227 * 1024);
    if (e != cudaSuccess) return e;
  }
  for (int q = 0; q < nprob; ++q) P.pdl |= probs[q].pdl;
  if (P.pdl) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(tiles * S);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_gemm_tc<false>, P);
    if (e != cudaSuccess) return e;
  } else {
    k_gemm_tc<false><<<tiles * S, kThreads, smem, s>>>(P);
  }
  return cudaGetLastError();
}

// Whether the tensor-core path takes a problem: TMA needs 16-byte aligned bases and row strides;
// grouped products need each group's K to be whole 64-wide slices.
bool gemm_tc_supported(const LinearProblem &q) {
  if (q.W8) {  // fp8 weights: 16-byte aligned codes and rows
    if (((uintptr_t)q.W8 & 15) || q.ldw % 16 || q.K % 16 || !q.w8_scale || ((uintptr_t)q.x & 15) || q.ldx % 8)
      return false;
    if (q.groups > 1 && q.K % (2 * gemm::BK)) return false;  // (a group's k-range is whole 128-wide units)
    return q.M > 0 && q.N > 0 && gemm::encoder() != nullptr;
  }
  if (((uintptr_t)q.x & 15) || ((uintptr_t)q.W & 15)) return false;
  if (q.ldx % 8 || q.ldw % 8 || q.K % 8) return false;
  if (q.groups > 1 && q.K % (gemm::BK * gemm::ATOMS)) return false;
  if (q.M <= 0 || q.N <= 0 || q.K <= 0) return false;
  return gemm::encoder() != nullptr;
}

}  // namespace csa

// ---- allocation-free projection -------------------------------------------------------------------
// csa_linear_noalloc: the same Stream-K product, for callers that cannot allocate device memory
// (an embedding runtime that owns a fixed device-memory budget, or code that runs without a
// csa_ctx, whose creation allocates workspaces).  Its scratch -- the arrival counters, the f32
// partials and a status word -- is this file-scope device array, which every GPU that loads the
// library holds until the process exits.  Host code must not hand the array's name to a kernel:
// in host code it is only a stand-in; the device address comes from cudaGetSymbolAddress, looked up
// by the first call made with a given device and CUDA context current (a device reset makes a new
// context, whose first call looks the address up again).

namespace csa {

// failure-detection test hook of the projection kernels on the current device (0: off)
cudaError_t set_gemm_stall(unsigned long long ns) { return cudaMemcpyToSymbol(gemm::g_stall_ns, &ns, sizeof(ns)); }

namespace {

constexpr int kNoAllocMaxM = 32;     // tokens: the partials below are sized for BN <= 32
constexpr int kNoAllocMaxGrid = 160;  // CTAs: one per SM on GB300 (152) with room to spare
constexpr size_t kNoAllocPartialBytes = (size_t)kNoAllocMaxGrid * 2 * gemm::BM * kNoAllocMaxM * sizeof(float);
constexpr size_t kNoAllocWsBytes = gemm::kCounterBytes + kNoAllocPartialBytes;
constexpr size_t kNoAllocBytes = kNoAllocWsBytes + 256;  // + the status word
constexpr int kNoAllocMaxDevices = 128;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
CtxGetCurrentFn ctx_get_current() {
  static const CtxGetCurrentFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(p);
    return static_cast<CtxGetCurrentFn>(nullptr);
  }();
  return fn;
}

std::mutex g_noalloc_mu;
struct NoAllocSlot {
  CUcontext ctx;  // the context the address belongs to
  void *addr;
  int sms;
};
NoAllocSlot g_noalloc[kNoAllocMaxDevices];

// The array's device address on the current device and context, looked up on first use there
// (under the lock, so concurrent first calls look it up once).  Returns CSA_OK or an error code.
int noalloc_scratch(const char *who, bool lookup, void **addr, int *sms) {
  *addr = nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(CSA_ERR_CUDA, "%s: cudaGetDevice: %s", who, cudaGetErrorString(e));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return set_error(CSA_ERR_ARG, "%s: device %d", who, dev);
  // the current context (NULL while the runtime has not made one current yet on this thread)
  CUcontext cur = nullptr;
  CtxGetCurrentFn get = ctx_get_current();
  if (!get || get(&cur) != CUDA_SUCCESS) return set_error(CSA_ERR_CUDA, "%s: cuCtxGetCurrent unavailable", who);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocSlot &sl = g_noalloc[dev];
  if (!cur || !sl.addr || sl.ctx != cur) {
    if (!lookup) return CSA_OK;  // nothing has run with this context
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // (makes the device's primary context current)
    if (e != cudaSuccess || !p) return set_error(CSA_ERR_CUDA, "%s: cudaGetSymbolAddress: %s", who, cudaGetErrorString(e));
    if (get(&cur) != CUDA_SUCCESS || !cur) return set_error(CSA_ERR_CUDA, "%s: no current context", who);
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return set_error(CSA_ERR_CUDA, "%s: device query: %s", who, cudaGetErrorString(e));
    sl.ctx = cur;
    sl.addr = p;
    sl.sms = n;
  }
  *addr = sl.addr;
  if (sms) *sms = sl.sms;
  return CSA_OK;
}

}  // namespace
}  // namespace csa

extern "C" int csa_linear_noalloc(const csa_bf16 *x, int M, int K, int ldx, const csa_bf16 *W, int N, int ldw,
                                  csa_bf16 *y, int ldy, int groups, csa_stream stream) {
  using namespace csa;
  if (!x || !W || !y) return set_error(CSA_ERR_ARG, "csa_linear_noalloc: NULL argument");
  if (M <= 0 || K <= 0 || N <= 0 || groups <= 0 || ldx < K * groups || ldw < K || ldy < N * groups)
    return set_error(CSA_ERR_ARG, "csa_linear_noalloc: bad shape M=%d K=%d N=%d groups=%d", M, K, N, groups);
  if (M > kNoAllocMaxM)
    return set_error(CSA_ERR_SHAPE, "csa_linear_noalloc: M=%d above the %d tokens its static scratch holds", M,
                     kNoAllocMaxM);
  const int64_t tiles = (int64_t)((N + gemm::BM - 1) / gemm::BM) * groups;
  if (tiles > gemm::kCounterInts)
    return set_error(CSA_ERR_SHAPE, "csa_linear_noalloc: %lld output tiles above %d", (long long)tiles,
                     gemm::kCounterInts);
  LinearProblem pr{(const bf16 *)x, M, K, ldx, (const bf16 *)W, N, ldw, (bf16 *)y, ldy, groups};
  if (!gemm_tc_supported(pr))
    return set_error(CSA_ERR_ARG,
                     "csa_linear_noalloc: operands and row strides must be 16-byte aligned, K a multiple of 8 "
                     "(of 64 with groups)");
  void *scratch = nullptr;
  int sms = 0;
  if (int rc = noalloc_scratch("csa_linear_noalloc", true, &scratch, &sms)) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  // the array keeps the last call's contents: the counters this launch uses must start at zero (the
  // status word is not cleared: it keeps a timeout until csa_linear_noalloc_status clears it)
  cudaError_t e = cudaMemsetAsync(scratch, 0, (size_t)tiles * sizeof(int), s);
  if (e != cudaSuccess) return set_error(CSA_ERR_CUDA, "csa_linear_noalloc: clear: %s", cudaGetErrorString(e));
  int *status = reinterpret_cast<int *>(static_cast<unsigned char *>(scratch) + kNoAllocWsBytes);
  e = launch_gemm_tc(&pr, 1, static_cast<float *>(scratch), kNoAllocWsBytes, std::min(sms, kNoAllocMaxGrid), status, s);
  if (e != cudaSuccess) return set_error(CSA_ERR_CUDA, "csa_linear_noalloc: launch: %s", cudaGetErrorString(e));
  return CSA_OK;
}

extern "C" int csa_linear_noalloc_status(int clear) {
  using namespace csa;
  void *scratch = nullptr;
  if (int rc = noalloc_scratch("csa_linear_noalloc_status", false, &scratch, nullptr)) return rc;
  if (!scratch) return CSA_OK;  // no call has run on this device and context
  int *status = reinterpret_cast<int *>(static_cast<unsigned char *>(scratch) + kNoAllocWsBytes);
  int st = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&st, status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(status, 0, sizeof(int));
  if (e == cudaSuccess && clear) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return set_error(CSA_ERR_CUDA, "csa_linear_noalloc_status: %s", cudaGetErrorString(e));
  if (st & kStatusTimeout) return set_error(CSA_ERR_DEVICE_TIMEOUT, "csa_linear_noalloc: a bounded device-side wait ran out");
  return CSA_OK;
}
