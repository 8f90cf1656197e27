// Tiered causal chunked-prefill attention on the 5th-generation tensor
// cores (tcgen05): one launch = (row block) x (device-resident cell range:
// the VRAM head or one arena bucket of the host tail).
//
// Per CTA: two query tiles A and B of 128 MMA rows each (128/G query
// positions x the G query heads of one kv head), against the whole cell range
// in tiles of 128 cells.
//   warps 0-3          : softmax + epilogue of tile A (thread = row = TMEM lane)
//   warps 4-7          : softmax + epilogue of tile B
//   warp 8             : producer, K and V tiles into separate 2-stage rings:
//                        device segments by TMA (one lane, two 64-dim SW128
//                        boxes per tile); host-memory segments (the tail read
//                        in place) by the 32 lanes with plain 16-byte loads
//                        stored in the same SW128 layout -- TMA never reads
//                        host memory
//   warp 9  (one lane) : MMA issuer; the warp owns the TMEM allocation.
//   warps 10-11        : bf16 caches only: each landed V tile rewritten in
//                        place as fp16 before its PV is issued
// TMEM: S_A, S_B (fp32, 128 columns each) and O_A, O_B (fp32, 128 each).
// The softmax writes P back over its S columns as fp16 (11 significant bits;
// P is in [0, 2^8]), and O += P V is issued once, both operands fp16, with P
// read from TMEM.  Issue order S_A S_B | PV_A S_A' PV_B S_B' | ... keeps the
// tensor core busy with one tile while the other tile's softmax runs.
// The running max is rescaled lazily (only when the tile max exceeds the
// reference by more than 2^8).  The running (m, l, acc) of earlier launches
// is folded in at the start and written back at the end (ExLlamaV3
// qsa-kv-offload patch, the fold of a bucket's partial into the running
// softmax), or the output normalised by max(l, 1e-30) on the last launch of
// a row block.
//
// Every mbarrier wait is bounded (about 2 s of %globaltimer); on timeout the
// waiter sets kErrWaitTimeout in the device error word and the CTA winds
// down, after the copies and MMAs it issued have landed.
#include <cuda.h>
#include <cstring>
#include <cuda_fp16.h>
#include <math.h>

#include "kvo_internal.cuh"
#include "sync.cuh"

namespace kvo {

namespace {

constexpr int BM = 128;                  // MMA rows per query tile
constexpr int NQ = 2;                    // query tiles per CTA
constexpr int BN = 128;                  // cells per tile
constexpr int HD = 128;                  // head dim
constexpr int kThreads = 384;            // warps 0-7 softmax, 8 TMA, 9 MMA, 10-11 V conversion
constexpr int kHalf = BM * 128;          // one SW128 half tile: 128 rows x 128 B = 16 KiB
constexpr int kTile = 2 * kHalf;         // 128 rows x 256 B
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;   // S_q at q*128, O_q at 256 + q*128
constexpr float kLazy = 8.0f;            // rescale when the max grows by > 2^8

// shared memory plan (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;                                 // NQ query tiles
constexpr int kOffK = kOffQ + NQ * kTile;                // kStages K tiles
constexpr int kOffV = kOffK + kStages * kTile;           // kStages V tiles
constexpr int kOffBar = kOffV + kStages * kTile;         // mbarriers + TMEM slot
constexpr int kSlack = 1024;                             // room to align the base to 1024 B
constexpr int kSmemBytes = kOffBar + 256 + kSlack;
static_assert(kSmemBytes <= 232448, "shared memory plan exceeds the per-CTA limit");

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// UMMA shared-memory descriptor, SW128 (layout type 2), version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16, fp32 accumulate, M = 128, N = 128.
template <int DT>
__host__ __device__ constexpr uint32_t idesc(bool b_mn_major) {
  return (1u << 4)                                   // D = f32
         | ((DT == KVO_BF16 ? 1u : 0u) << 7)         // A type
         | ((DT == KVO_BF16 ? 1u : 0u) << 10)        // B type
         | ((b_mn_major ? 1u : 0u) << 16)            // B major
         | ((uint32_t)(BN >> 3) << 17)               // N
         | ((uint32_t)(BM >> 4) << 24);              // M
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                     uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accum));
}

// As umma, with matrix A read from TMEM (M lanes x K columns of packed pairs).
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id,
                                        uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(accum));
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.  The load and its
// wait are one asm statement, so no use of the registers can be scheduled
// before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// All 128 fp32 columns of this thread's TMEM lane in one load and one wait
// (one round trip for the whole S row).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float *v) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
      "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,"
      "%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,"
      "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]),"=r"(r[1]),"=r"(r[2]),"=r"(r[3]),"=r"(r[4]),"=r"(r[5]),"=r"(r[6]),"=r"(r[7]),"=r"(r[8]),"=r"(r[9]),"=r"(r[10]),"=r"(r[11]),"=r"(r[12]),"=r"(r[13]),"=r"(r[14]),"=r"(r[15]),
        "=r"(r[16]),"=r"(r[17]),"=r"(r[18]),"=r"(r[19]),"=r"(r[20]),"=r"(r[21]),"=r"(r[22]),"=r"(r[23]),"=r"(r[24]),"=r"(r[25]),"=r"(r[26]),"=r"(r[27]),"=r"(r[28]),"=r"(r[29]),"=r"(r[30]),"=r"(r[31]),
        "=r"(r[32]),"=r"(r[33]),"=r"(r[34]),"=r"(r[35]),"=r"(r[36]),"=r"(r[37]),"=r"(r[38]),"=r"(r[39]),"=r"(r[40]),"=r"(r[41]),"=r"(r[42]),"=r"(r[43]),"=r"(r[44]),"=r"(r[45]),"=r"(r[46]),"=r"(r[47]),
        "=r"(r[48]),"=r"(r[49]),"=r"(r[50]),"=r"(r[51]),"=r"(r[52]),"=r"(r[53]),"=r"(r[54]),"=r"(r[55]),"=r"(r[56]),"=r"(r[57]),"=r"(r[58]),"=r"(r[59]),"=r"(r[60]),"=r"(r[61]),"=r"(r[62]),"=r"(r[63]),
        "=r"(r[64]),"=r"(r[65]),"=r"(r[66]),"=r"(r[67]),"=r"(r[68]),"=r"(r[69]),"=r"(r[70]),"=r"(r[71]),"=r"(r[72]),"=r"(r[73]),"=r"(r[74]),"=r"(r[75]),"=r"(r[76]),"=r"(r[77]),"=r"(r[78]),"=r"(r[79]),
        "=r"(r[80]),"=r"(r[81]),"=r"(r[82]),"=r"(r[83]),"=r"(r[84]),"=r"(r[85]),"=r"(r[86]),"=r"(r[87]),"=r"(r[88]),"=r"(r[89]),"=r"(r[90]),"=r"(r[91]),"=r"(r[92]),"=r"(r[93]),"=r"(r[94]),"=r"(r[95]),
        "=r"(r[96]),"=r"(r[97]),"=r"(r[98]),"=r"(r[99]),"=r"(r[100]),"=r"(r[101]),"=r"(r[102]),"=r"(r[103]),"=r"(r[104]),"=r"(r[105]),"=r"(r[106]),"=r"(r[107]),"=r"(r[108]),"=r"(r[109]),"=r"(r[110]),"=r"(r[111]),
        "=r"(r[112]),"=r"(r[113]),"=r"(r[114]),"=r"(r[115]),"=r"(r[116]),"=r"(r[117]),"=r"(r[118]),"=r"(r[119]),"=r"(r[120]),"=r"(r[121]),"=r"(r[122]),"=r"(r[123]),"=r"(r[124]),"=r"(r[125]),"=r"(r[126]),"=r"(r[127])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Packed fp32 pairs (low word = first element).
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float &a, float &b) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
      "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
      "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

template <int DT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (DT == KVO_BF16) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 2^x on the SFU (PTX ex2.approx.ftz.f32; 2^-inf = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two bf16 values (one word) -> the same two values as fp16, rounded to
// nearest (bf16 -> fp32 is exact: the bits shifted up).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack2<KVO_F16>(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Byte offset of 16-byte chunk c (0..15 across the 256-byte row) of row r in
// a tile made of two SW128 halves of [128 rows][128 B].
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)((c >> 3) * kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

struct TcParams {
  PrefillArgs a;
  uint32_t *err;
  // non-null: the segment's K/V rows are host memory, row (c - a.hi_origin)
  // at host_k / host_v (the tensor maps are unused)
  const uint8_t *host_k, *host_v;
};

// Host-memory producer: the 128 cell rows [t0, t0 + 128) of kv head g into a
// tile of two SW128 halves, 16-byte loads kHostBatch at a time per lane;
// rows at or past c_end are zero (finite values for the masked PV).
constexpr int kHostBatch = 16;

__device__ __forceinline__ void host_tile(const uint8_t *base, int64_t row_bytes, int64_t hi_origin, int g,
                                          int64_t t0, int64_t c_end, uint8_t *dst, int lane) {
  constexpr int kChunks = BN * 16;                   // 16-byte chunks of the tile (256 B per row)
  for (int i0 = 0; i0 < kChunks; i0 += 32 * kHostBatch) {
    int4 v[kHostBatch];
#pragma unroll
    for (int u = 0; u < kHostBatch; ++u) {
      const int i = i0 + u * 32 + lane, r = i >> 4, c = i & 15;
      const int64_t cell = t0 + r;
      v[u] = cell < c_end ? *((const int4 *)(base + (cell - hi_origin) * row_bytes + g * (HD * 2)) + c)
                          : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kHostBatch; ++u) {
      const int i = i0 + u * 32 + lane, r = i >> 4, c = i & 15;
      *(int4 *)(dst + sw128(r, c)) = v[u];
    }
  }
}

template <int DT, int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const TcParams P) {
  constexpr int PB = BM / G;                         // query positions per tile
  const PrefillArgs &a = P.a;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // SW128 tiles want a 1024-byte aligned base; the slack covers the
  // misalignment, beyond which the CTA reports and exits.
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad > (uint32_t)(kSlack - 256)) {
    if (threadIdx.x == 0) atomicOr(P.err, kErrSmemAlign);
    return;
  }
  uint8_t *smem = smem_raw + pad;
  uint64_t *bar = (uint64_t *)(smem + kOffBar);
  uint64_t *full_k = bar;                  // [kStages] TMA -> MMA
  uint64_t *empty_k = bar + 2;             // [kStages] MMA -> TMA
  uint64_t *full_v = bar + 4;
  uint64_t *empty_v = bar + 6;
  uint64_t *s_full = bar + 8;              // [NQ] MMA -> softmax (S of tile q ready)
  uint64_t *p_full = bar + 10;             // [NQ] softmax -> MMA (128 arrivals)
  uint64_t *o_done = bar + 12;             // [NQ] MMA -> softmax (PV of tile q finished)
  uint64_t *fin = bar + 14;                // MMA teardown
  uint64_t *conv_v = bar + 16;             // [kStages] converters -> MMA (bf16: V tile now fp16)
  uint32_t *tmem_slot = (uint32_t *)(bar + 18);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y;
  const int i0 = blockIdx.x * (NQ * PB);             // first query row of the CTA
  const int n_pos = a.rows - i0 < NQ * PB ? a.rows - i0 : NQ * PB;
  const int64_t cta_last = a.pos0 + i0 + n_pos - 1;
  const int64_t c_end = a.c1 < cta_last + 1 ? a.c1 : cta_last + 1;
  const int n_tiles = c_end > a.c0 ? (int)((c_end - a.c0 + BN - 1) / BN) : 0;

  if (tid == 0) {
    for (int i = 0; i < 14; ++i) mbar_init(&bar[i], (i == 10 || i == 11) ? BM : 1);
    mbar_init(fin, 1);
    for (int s = 0; s < kStages; ++s) mbar_init(&conv_v[s], 2);   // one arrival per converter warp
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Query tiles (all threads): row r of tile q = position q*PB + r/G, head g*G + r%G.
  // Loads go out kQBatch at a time per thread, so that their latencies overlap.
  constexpr int kQChunks = NQ * BM * 16, kQBatch = 8;
  for (int j0 = tid; j0 < kQChunks; j0 += kThreads * kQBatch) {
    int4 v[kQBatch];
#pragma unroll
    for (int u = 0; u < kQBatch; ++u) {
      const int i = j0 + u * kThreads;
      const int q = i / (BM * 16), rr = (i >> 4) % BM, c = i & 15;
      const int pi = q * PB + rr / G, hh = rr % G;
      v[u] = make_int4(0, 0, 0, 0);
      if (i < kQChunks && pi < n_pos)
        v[u] = *((const int4 *)(a.q + ((size_t)(i0 + pi) * a.n_q_heads + g * G + hh) * HD) + c);
    }
#pragma unroll
    for (int u = 0; u < kQBatch; ++u) {
      const int i = j0 + u * kThreads;
      const int q = i / (BM * 16), rr = (i >> 4) % BM, c = i & 15;
      if (i < kQChunks) *(int4 *)(smem + kOffQ + q * kTile + sw128(rr, c)) = v[u];
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // Q visible to the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Registers: the block starts at 168 a thread (384 x 168 = 64,512).  Warps
  // 8-11 (producer, MMA issuer, converters) hand theirs down to 136 and the
  // two softmax warpgroups take 184 each: 2 x 128 x 184 + 128 x 136 = 64,512,
  // the launch's own total, so the increase is always satisfied (and the
  // softmax keeps its whole S row in registers without spilling).
  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 136;" ::: "memory");
  if (warp == 8 && P.host_k) {
    // ---------------------------------------------------------------- host-memory producer
    // The 32 lanes fill each K and V stage with plain loads; after its stores
    // every lane fences them into the async proxy, then lane 0 arrives on the
    // stage's full barrier (nothing is in flight between tiles, so a failed
    // wait leaves no copy to drain).
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int s = j % kStages;
      const int64_t t0 = a.c0 + (int64_t)j * BN;
      if (j >= kStages) ok = __all_sync(0xffffffffu, mbar_wait(&empty_k[s], ((j / kStages) - 1) & 1, P.err));
      if (!ok) break;
      host_tile(P.host_k, a.row_bytes, a.hi_origin, g, t0, c_end, smem + kOffK + s * kTile, lane);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&full_k[s]);
      if (j >= kStages) ok = __all_sync(0xffffffffu, mbar_wait(&empty_v[s], ((j / kStages) - 1) & 1, P.err));
      if (!ok) break;
      host_tile(P.host_v, a.row_bytes, a.hi_origin, g, t0, c_end, smem + kOffV + s * kTile, lane);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&full_v[s]);
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && n_tiles > 0) {
      bool ok = true;
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int s = j % kStages;
        const int y = (int)(a.c0 + (int64_t)j * BN - a.hi_origin);   // row in the segment map
        if (j >= kStages) ok = mbar_wait(&empty_k[s], ((j / kStages) - 1) & 1, P.err);
        if (!ok) break;
        mbar_expect_tx(&full_k[s], kTile);
        uint8_t *kd = smem + kOffK + s * kTile;
        tma_load_2d(kd, &tmap_k, g * HD, y, &full_k[s]);
        tma_load_2d(kd + kHalf, &tmap_k, g * HD + 64, y, &full_k[s]);
        issued_k = j + 1;
        if (j >= kStages) ok = mbar_wait(&empty_v[s], ((j / kStages) - 1) & 1, P.err);
        if (!ok) break;
        mbar_expect_tx(&full_v[s], kTile);
        uint8_t *vd = smem + kOffV + s * kTile;
        tma_load_2d(vd, &tmap_v, g * HD, y, &full_v[s]);
        tma_load_2d(vd + kHalf, &tmap_v, g * HD + 64, y, &full_v[s]);
        issued_v = j + 1;
      }
      if (!ok) {
        // let the copies already issued land before the CTA exits
        for (int j = issued_k - kStages < 0 ? 0 : issued_k - kStages; j < issued_k; ++j)
          mbar_wait(&full_k[j % kStages], (j / kStages) & 1, P.err);
        for (int j = issued_v - kStages < 0 ? 0 : issued_v - kStages; j < issued_v; ++j)
          mbar_wait(&full_v[j % kStages], (j / kStages) & 1, P.err);
      }
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t id_s = idesc<DT>(false);
      constexpr uint32_t id_o = idesc<KVO_F16>(true);       // P and V both fp16
      // V tile ready for PV: landed (fp16 caches) or converted (bf16 caches)
      uint64_t *ready_v = DT == KVO_BF16 ? conv_v : full_v;
      uint32_t o_acc = a.init ? 0u : 1u;
      bool ok = true;
      // S_q(j) = Q_q K_j^T into the S columns of tile q
      auto issue_s = [&](int q, int j) {
        const uint32_t q_base = smem_u32(smem + kOffQ + q * kTile);
        const uint32_t k_base = smem_u32(smem + kOffK + (j % kStages) * kTile);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kHalf + (ks & 3) * 32;
          umma(tmem + kColS + q * 128, sdesc(q_base + off, 16, 1024), sdesc(k_base + off, 16, 1024),
               id_s, ks > 0);
        }
        umma_commit(&s_full[q]);
      };
      // O_q += P_q V_j with P_q (fp16 pairs over the S columns) read from TMEM
      auto issue_pv = [&](int q, int j) {
        const uint32_t v_base = smem_u32(smem + kOffV + (j % kStages) * kTile);
        const uint32_t d_o = tmem + kColO + q * 128;
        // cells 16kk..16kk+15: the pairs in columns 8kk..8kk+7
        const uint32_t p_base = tmem + kColS + q * 128;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bd = sdesc(v_base + kk * 16 * 128, kHalf, 1024);
          umma_ts(d_o, p_base + 8 * kk, bd, id_o, (kk > 0) || o_acc);
        }
        umma_commit(&o_done[q]);
      };
      ok = mbar_wait(&full_k[0], 0, P.err);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
        umma_commit(&empty_k[0]);
      }
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int jn = j + 1;
        ok = mbar_wait(&ready_v[j % kStages], (j / kStages) & 1, P.err);
        if (!ok) break;
        ok = mbar_wait(&p_full[0], j & 1, P.err);
        if (!ok) break;
        tc_fence_after();
        issue_pv(0, j);
        if (jn < n_tiles) {
          ok = mbar_wait(&full_k[jn % kStages], (jn / kStages) & 1, P.err);
          if (!ok) break;
          tc_fence_after();
          issue_s(0, jn);
        }
        ok = mbar_wait(&p_full[1], j & 1, P.err);
        if (!ok) break;
        tc_fence_after();
        issue_pv(1, j);
        o_acc = 1u;
        umma_commit(&empty_v[j % kStages]);
        if (jn < n_tiles) {
          issue_s(1, jn);
          umma_commit(&empty_k[jn % kStages]);
        }
      }
      // all issued tensor-core work has finished once this arrives
      umma_commit(fin);
      mbar_wait(fin, 0, P.err);
    }
  } else if (warp >= 10) {
    // ---------------------------------------------------------------- V conversion (bf16)
    // Each landed V tile is rewritten in place as fp16 (the swizzle moves
    // whole 16-byte chunks, so only the values change), fenced into the async
    // proxy and handed to the MMA warp.  bf16 -> fp16 is exact for magnitudes
    // in [2^-14, 65504]; smaller ones round to fp16's subnormal grid (absolute
    // error <= 2^-25); one that becomes infinite (65520 and above, or an
    // infinite input) sets kErrF16Range.
    if constexpr (DT == KVO_BF16) {
      constexpr int kChunks = kTile / 16, kLanes = 64, kBatch = 8;
      const int cl = (warp - 10) * 32 + lane;
      __half2 vmax = __float2half2_rn(0.f);                   // max |v| as fp16
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int s = j % kStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&full_v[s], (j / kStages) & 1, P.err));
        if (!ok) break;
        uint4 *vt = (uint4 *)(smem + kOffV + s * kTile);
#pragma unroll 1
        for (int i0 = cl; i0 < kChunks; i0 += kLanes * kBatch) {
          uint4 u[kBatch];
#pragma unroll
          for (int k = 0; k < kBatch; ++k) u[k] = vt[i0 + k * kLanes];
#pragma unroll
          for (int k = 0; k < kBatch; ++k) {
            u[k].x = bf16x2_to_f16x2(u[k].x);
            u[k].y = bf16x2_to_f16x2(u[k].y);
            u[k].z = bf16x2_to_f16x2(u[k].z);
            u[k].w = bf16x2_to_f16x2(u[k].w);
            const __half2 m01 = __hmax2(__habs2(*(const __half2 *)&u[k].x), __habs2(*(const __half2 *)&u[k].y));
            const __half2 m23 = __hmax2(__habs2(*(const __half2 *)&u[k].z), __habs2(*(const __half2 *)&u[k].w));
            vmax = __hmax2(vmax, __hmax2(m01, m23));
          }
#pragma unroll
          for (int k = 0; k < kBatch; ++k) vt[i0 + k * kLanes] = u[k];
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&conv_v[s]);
      }
      const uint32_t mb = *(const uint32_t *)&vmax;
      if ((mb & 0x7fffu) >= 0x7c00u || ((mb >> 16) & 0x7fffu) >= 0x7c00u) atomicOr(P.err, kErrF16Range);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;" ::: "memory");
    // ---------------------------------------------------------------- softmax + epilogue
    const int q = warp >> 2;                                  // query tile
    const int r = (warp & 3) * 32 + lane;                     // row = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_addr = lane_addr + kColS + q * 128;
    const uint32_t o_addr = lane_addr + kColO + q * 128;
    const int pi = q * PB + r / G;
    const bool row_ok = pi < n_pos;
    const int64_t pos = a.pos0 + i0 + pi;
    const size_t row_idx = (size_t)(i0 + pi) * a.n_q_heads + g * G + (r % G);
    float m_used = -INFINITY, l = 0.f;
    bool o_valid = !a.init;                                   // O holds data (from the state)
    if (!a.init && row_ok) {
      m_used = a.ml[row_idx * 2];
      l = a.ml[row_idx * 2 + 1];
    }
    if (!a.init) {
      // load the running accumulator into TMEM (rows past the launch get zeros),
      // 64 columns' loads in flight at a time
      float v[64];
#pragma unroll
      for (int c = 0; c < 4; c += 2) {
#pragma unroll
        for (int i = 0; i < 64; i += 4) {
          float4 x = row_ok ? *(const float4 *)(a.acc + row_idx * HD + c * 32 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[i] = x.x; v[i + 1] = x.y; v[i + 2] = x.z; v[i + 3] = x.w;
        }
        tmem_st32(o_addr + c * 32, v);
        tmem_st32(o_addr + (c + 1) * 32, v + 32);
      }
      tmem_wait_st();
    }
    tc_fence_before();
    // first position of this tile's rows: cells at or before it are visible to all of them
    const int64_t first_pos = a.pos0 + i0 + q * PB;
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[q], j & 1, P.err));
      if (!ok) break;
      tc_fence_after();
      const int64_t t0 = a.c0 + (int64_t)j * BN;
      const bool need_mask = (t0 + BN > c_end) || (t0 + BN - 1 > first_pos) || !row_ok;
      // The whole S row of this thread in registers: one TMEM round trip.
      // Row max of the raw scores (scale > 0), 8 chains of 3-input maxima.
      float x[BN];
      tmem_ld128(s_addr, x);
      if (need_mask) {
#pragma unroll
        for (int i = 0; i < BN; ++i) {
          const int64_t cj = t0 + i;
          if (!row_ok || cj >= c_end || cj > pos) x[i] = -INFINITY;
        }
      }
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
#pragma unroll
      for (int i = 0; i < BN; i += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = max3(mx[k], x[i + 2 * k], x[i + 2 * k + 1]);
      const float mt = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) *
                       a.scale_log2;
      // Lazy rescale (warp-uniform: tcgen05.ld/st are warp-collective): a row
      // whose tile max exceeds its reference by more than 2^8 moves its
      // reference to the tile max and rescales l and O by 2^(old - new).
      const bool mine = mt > m_used + kLazy;
      float alpha = 1.f;
      if (mine) alpha = m_used == -INFINITY ? 0.f : exp2f(m_used - mt);
      const bool rescale = __any_sync(0xffffffffu, mine);
      if (rescale) l *= alpha;
      if (mine) m_used = mt;
      const float nref = m_used == -INFINITY ? 0.f : -m_used;
      // P = 2^(s*scale - ref) from the registers (a masked score is -inf and
      // gives +0), written back as fp16 over the S columns it came from: cells
      // 2k, 2k+1 -> column k.  The PV of the previous tile read these columns
      // before this tile's S was written into them.  Arguments and sums run
      // as packed fp32 pairs; l sums the unrounded p.
      const uint64_t sc2 = pk2(a.scale_log2, a.scale_log2), nr2 = pk2(nref, nref);
      uint64_t sm2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float a0, a1;
          upk2(ffma2(pk2(x[64 * c + 2 * e], x[64 * c + 2 * e + 1]), sc2, nr2), a0, a1);
          const float p0 = ex2(a0), p1 = ex2(a1);
          sm2[e & 3] = fadd2(sm2[e & 3], pk2(p0, p1));
          w[e] = pack2<KVO_F16>(p0, p1);
        }
        tmem_st32u(s_addr + c * 32, w);
      }
      {
        float u0, u1, u2, u3, u4, u5, u6, u7;
        upk2(sm2[0], u0, u1);
        upk2(sm2[1], u2, u3);
        upk2(sm2[2], u4, u5);
        upk2(sm2[3], u6, u7);
        l += ((u0 + u2) + (u4 + u6)) + ((u1 + u3) + (u5 + u7));
      }
      tmem_wait_st();
      // O follows a moved reference (after P, so that S no longer occupies
      // registers): wait until the previous tile's PV has finished with it.
      if (rescale && o_valid) {
        if (j > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&o_done[q], (j - 1) & 1, P.err));
          if (!ok) break;
          tc_fence_after();
        }
        float v[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tmem_ld32(o_addr + c * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= alpha;
          tmem_st32(o_addr + c * 32, v);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(&p_full[q]);
      o_valid = true;
    }
    // ---- epilogue: wait for the last PV, then write state or output
    if (ok && n_tiles > 0) ok = __all_sync(0xffffffffu, mbar_wait(&o_done[q], (n_tiles - 1) & 1, P.err));
    tc_fence_after();
    if (ok) {
      const float inv = a.finalize ? 1.f / fmaxf(l, 1e-30f) : 1.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        if (o_valid) {                                       // warp-uniform
          tmem_ld32(o_addr + c * 32, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *(float4 *)(a.acc + row_idx * HD + c * 32 + i) =
                make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv);
        }
      }
      if (!a.finalize && row_ok) {
        a.ml[row_idx * 2] = m_used;
        a.ml[row_idx * 2 + 1] = l;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
    else
      cudaGetLastError();
  }
  return fn;
}

// 2D map over [rows][n_kv_heads * 128] elements, boxes of [128 rows][64 elems], SW128.
int make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t row_bytes, int dt) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(KVO_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {64, (cuuint32_t)BN};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt == KVO_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                  const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KVO_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return KVO_OK;
}

template <int DT, int G>
cudaError_t launch_g(const CUtensorMap &mk, const CUtensorMap &mv, const TcParams &p, cudaStream_t st) {
  constexpr int PB = NQ * BM / G;                    // query positions per CTA
  auto k = prefill_tc_kernel<DT, G>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((p.a.rows + PB - 1) / PB, p.a.n_kv_heads);
  k<<<grid, kThreads, kSmemBytes, st>>>(mk, mv, p);
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dt(const CUtensorMap &mk, const CUtensorMap &mv, const TcParams &p, cudaStream_t st) {
  switch (p.a.group) {
    case 1: return launch_g<DT, 1>(mk, mv, p, st);
    case 2: return launch_g<DT, 2>(mk, mv, p, st);
    case 4: return launch_g<DT, 4>(mk, mv, p, st);
    default: return launch_g<DT, 8>(mk, mv, p, st);
  }
}

}  // namespace

// Launch over a host-memory segment (the tail read in place): cells [a.c0,
// a.c1) are rows (c - a.hi_origin) of a.k_hi / a.v_hi, loaded by the producer
// warp with plain loads.
int launch_prefill_tc_host(const PrefillArgs &a, cudaStream_t st) {
  CUtensorMap unused;
  memset(&unused, 0, sizeof(unused));
  TcParams p;
  p.a = a;
  p.err = device_error_word();
  if (!p.err) return fail(KVO_ERR_CUDA, "device error word unavailable");
  p.host_k = a.k_hi;
  p.host_v = a.v_hi;
  cudaError_t e = a.dtype == KVO_BF16 ? launch_dt<KVO_BF16>(unused, unused, p, st)
                                      : launch_dt<KVO_F16>(unused, unused, p, st);
  return cuda_status(e, "tcgen05 prefill launch (host segment)");
}

// Launch over a device-resident segment: cells [a.c0, a.c1) are rows
// (c - a.hi_origin) of the buffers k_seg / v_seg, which hold seg_rows rows.
int launch_prefill_tc(const PrefillArgs &a, const void *k_seg, const void *v_seg, int64_t seg_rows,
                      cudaStream_t st) {
  CUtensorMap mk, mv;
  const int64_t cols = (int64_t)a.n_kv_heads * HD;
  int r = make_map(&mk, k_seg, seg_rows, cols, a.row_bytes, a.dtype);
  if (r) return r;
  r = make_map(&mv, v_seg, seg_rows, cols, a.row_bytes, a.dtype);
  if (r) return r;
  TcParams p;
  p.a = a;
  p.err = device_error_word();
  if (!p.err) return fail(KVO_ERR_CUDA, "device error word unavailable");
  p.host_k = p.host_v = nullptr;
  cudaError_t e = a.dtype == KVO_BF16 ? launch_dt<KVO_BF16>(mk, mv, p, st) : launch_dt<KVO_F16>(mk, mv, p, st);
  return cuda_status(e, "tcgen05 prefill launch");
}

}  // namespace kvo
