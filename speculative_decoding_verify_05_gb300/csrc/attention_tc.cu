// Verify attention on tcgen05 tensor cores: persistent, stream-K over key tiles.
//
// Work: for every (sequence b, kv head h) the R = G * (gamma_b + 1) <= 64 query
// rows of the group attend keys 0 .. ctx_b + gamma_b under the causal rule
// "row j sees keys <= ctx_b + j / G".  The keys of all (b, h) pairs are cut
// into 128-key tiles and concatenated (b-major, then h); one CTA per SM takes
// an equal contiguous range of tiles, so every SM streams the same number of
// K/V bytes whatever the context lengths.  A range covers whole (b, h) pairs
// and at most two partial ones; a partial pair's unnormalised output (O,
// running max, running sum) goes to the workspace and the CTA that arrives
// last on the pair's counter merges the pieces in CTA order (no waiting).
//
// Per tile:
//   S[row, key] = Q . K_tile^T     tcgen05.mma M = 64 rows, N = 128 keys, K = 128 dims
//   softmax: an M = 64 accumulator keeps row r in TMEM lane (r / 16) * 32 + r % 16;
//            a split TMEM load (.16x32bx2) hands keys 0-63 of those 16 lanes to one
//            half-warp and keys 64-127 to the other, so two threads share a row: row
//            max, exp2 and row sum stay in registers (one shuffle each) and the P row
//            goes straight to shared memory
//   O[row, d] += P . V_tile        tcgen05.mma M = 64, N = 128 dims (V read MN-major), K = 128 keys
// Roles (8 warps): 0-3 softmax + epilogue; 4 and 6 only issue the TMA loads of K
// (2-stage ring) and V (4-stage ring: a V tile waits for the softmax, a K tile only for
// QK^T); 5 issues the MMAs (lane 0, event driven: whichever of QK^T or PV has its inputs
// ready goes first); 7 stages each pair's Q rows and patches the newest gamma_b + 1 keys
// (from Knew) into the K tiles holding keys >= ctx once their loads land; the softmax
// warps do the same for V (zeroing the rows past the block) just before that tile's PV.
// Both write the new rows into the cache too.  S and O are double buffered, Q and P single:
// shared memory goes to the K/V rings instead, whose depth sets the bytes each SM keeps in
// flight (for the same reason the per-sequence metadata sits in the V ring during the setup
// only, and in global memory afterwards).
#include "common.cuh"
#include "internal.h"

namespace spec {
namespace {

constexpr int D = 128;
constexpr int KT = 128;                  // keys per tile = MMA N of QK^T, MMA K of PV
constexpr int QR = 64;                   // query rows per (b, h) pair = MMA M
// Ring depths and Q buffers, measured on the 64-sequence verify launch (K/V stages, Q buffers:
// time): 2/3/2 203 us with the metadata resident in shared memory; 2/4/1 191 us, 3/3/1 197 us,
// 2/3/1 194 us with it in the V ring during the setup only.
constexpr int ST_K = 2;                  // K ring stages
constexpr int ST_V = 4;                  // V ring stages
constexpr int QB = 1;                    // Q buffers
constexpr int KV_HALF = KT * 128;        // 128 keys x 64 dims (128 B rows), 16 KB
constexpr int KV_TILE = 2 * KV_HALF;     // 32 KB
constexpr int Q_HALF = QR * 128;         // 64 rows x 64 bf16, 8 KB
constexpr int THREADS = 256;
constexpr uint32_t TMEM_COLS = 512;      // S x2 then O x2, 128 columns each
constexpr int MAX_B = 1024;              // sequences per call handled by this kernel

constexpr int OFF_K = 0;
constexpr int OFF_V = ST_K * KV_TILE;
constexpr int OFF_Q = OFF_V + ST_V * KV_TILE;       // QB buffers x two 64-dim halves
constexpr int OFF_P = OFF_Q + QB * 2 * Q_HALF;      // [64 rows][128 keys] as two 64-key halves
constexpr int OFF_BAR = OFF_P + 2 * Q_HALF;
constexpr int N_BARS = 3 * (ST_K + ST_V) + 8 + 2 * QB;
static_assert((N_BARS + 4) * 8 <= 256, "barrier block");
constexpr int OFF_FLAG = OFF_BAR + 256;             // merge flag, then the first cursor
constexpr int SMEM = OFF_FLAG + 64 + 1024;          // + alignment slack
// the setup keeps ctx, cu_rows and the unit prefix (3 B + 2 ints) in the V ring before its first load
static_assert(3 * MAX_B + 2 <= ST_V * KV_TILE / 4, "setup metadata");
static_assert(SMEM <= 227 * 1024, "shared memory budget");

// Non-blocking probe of an mbarrier phase (the event-driven MMA loop polls several barriers).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void bar_compute() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// 2^x on the special-function unit (ex2.approx: relative error ~2^-22; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory descriptor of an MN-major operand stored as 128-byte swizzled
// rows (8-row atoms 1024 B apart along K; 64-element atom columns `lbo` apart along M/N).
__device__ __forceinline__ uint64_t umma_desc_sw128_mn(uint32_t smem_addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= uint64_t((smem_addr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t(1024 >> 4) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 TMEM lanes, 128 columns split between the half-warps: threads 0-15 get columns
// [c, c + 64) of lanes base .. base + 15, threads 16-31 columns [c + 64, c + 128) of the same
// lanes (one asm with its wait, so no register is read before the load completes).
__device__ __forceinline__ void tmem_ld_split64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64+0], 64;\n"
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64+32], 64;\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
// The matching store of 16 columns per half-warp (columns [c, c + 16) and [c + 64, c + 80)).
__device__ __forceinline__ void tmem_st_split16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], 64, {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}

// Per-sequence metadata: during the setup a copy in shared memory (the V ring, idle until the
// first load), afterwards the caller's arrays and the CTA's own prefix slice of the workspace.
struct Meta {
  const int* pfx;   // [B + 1] first unit of sequence b (pfx[B] = total units)
  const int* ctx;   // [B] cached context length
  const int* cu;    // [B + 1] verify-row offsets
};

// Walks the tile list: unit u = (sequence b, kv head h, tile t).
struct Cursor {
  long long u;
  int b, h, t, nt, ctx, r0, Mb;
};
__device__ __forceinline__ void cur_seq(Cursor& c, const Meta& m, int B) {
  if (c.b < B) {
    c.ctx = m.ctx[c.b];
    c.r0 = m.cu[c.b];
    c.Mb = m.cu[c.b + 1] - c.r0;
    c.nt = (c.ctx + c.Mb + KT - 1) / KT;
  }
}
__device__ __forceinline__ Cursor cur_at(const Meta& m, int B, long long u) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (m.pfx[mid] <= u) lo = mid; else hi = mid - 1;
  }
  Cursor c;
  c.u = u;
  c.b = lo;
  cur_seq(c, m, B);
  const int rem = (int)(u - m.pfx[lo]);
  c.h = rem / c.nt;
  c.t = rem - c.h * c.nt;
  return c;
}
__device__ __forceinline__ void cur_next(Cursor& c, const Meta& m, int B, int Hkv) {
  ++c.u;
  if (++c.t == c.nt) {
    c.t = 0;
    if (++c.h == Hkv) {
      c.h = 0;
      ++c.b;
      cur_seq(c, m, B);
    }
  }
}

// Cost-balanced split of the tile list: a tile costs WT, starting a pair costs wp more, so
// unit u of pair p = b Hkv + h ends at cumulative cost C(u) = WT (u + 1) + wp (p + 1) and CTA
// c owns the units with floor((C(u) - 1) grid / Ctot) == c.  CTAs that cover many short
// pairs (each with its own epilogue, tail patch and possibly a merge) get fewer tiles.
constexpr long long WT = 4;
struct Part {
  long long U, Ctot;   // units, total cost
  int P, grid, Hkv, wp;
};
__device__ __forceinline__ long long cost_end(const Part& q, long long u, int p) {
  return WT * (u + 1) + (long long)q.wp * (p + 1);
}
__device__ __forceinline__ int cta_of(const Part& q, long long u, int p) {
  const long long c = (cost_end(q, u, p) - 1) * q.grid / q.Ctot;
  return c < q.grid - 1 ? (int)c : q.grid - 1;
}
// first unit of pair p; nt = its tiles
__device__ __forceinline__ long long pair_first(const Meta& m, int Hkv, int p, int& nt) {
  const int b = p / Hkv, h = p - b * Hkv;
  nt = (m.ctx[b] + m.cu[b + 1] - m.cu[b] + KT - 1) / KT;
  return m.pfx[b] + (long long)h * nt;
}
// first unit owned by CTA c (U for c >= grid): the smallest u with C(u) >= T(c)
__device__ long long range_start(const Part& q, const Meta& m, int c) {
  if (c <= 0 || q.U == 0) return 0;
  if (c >= q.grid) return q.U;
  const long long T = ((long long)c * q.Ctot + q.grid - 1) / q.grid + 1;
  if (T > q.Ctot) return q.U;             // more CTAs than cost units: this one and the rest are empty
  int lo = 0, hi = q.P - 1, nt;
  while (lo < hi) {                       // first pair whose last unit reaches T (C(U - 1) = Ctot)
    const int mid = (lo + hi) >> 1;
    const long long f = pair_first(m, q.Hkv, mid, nt);
    if (cost_end(q, f + nt - 1, mid) >= T) hi = mid; else lo = mid + 1;
  }
  const long long f = pair_first(m, q.Hkv, lo, nt);
  const long long need = T - (long long)q.wp * (lo + 1);    // WT (u + 1) >= need
  long long t = (need > 0 ? (need + WT - 1) / WT : 0) - 1 - f;
  t = t < 0 ? 0 : (t > nt - 1 ? nt - 1 : t);
  return f + t;
}

// 64 consecutive outputs v[d] * f rounded to bf16 (eight 16-byte stores).
__device__ __forceinline__ void store_half_bf16(uint16_t* dst, const float* v, float f) {
#pragma unroll
  for (int d = 0; d < 64; d += 8)
    *reinterpret_cast<uint4*>(dst + d) =
        make_uint4(pack_bf16x2(v[d] * f, v[d + 1] * f), pack_bf16x2(v[d + 2] * f, v[d + 3] * f),
                   pack_bf16x2(v[d + 4] * f, v[d + 5] * f), pack_bf16x2(v[d + 6] * f, v[d + 7] * f));
}

// A tile holding keys >= ctx (the last one or two of a pair): its rows rr0 .. rr0 + n_new - 1
// are keys first_new .. first_new + n_new - 1 of the new block.
struct TailRows {
  int rr0, n_new, first_new;
};
__device__ __forceinline__ TailRows tail_rows(const Cursor& c) {
  const int key0 = c.t * KT;
  TailRows g;
  g.rr0 = c.ctx > key0 ? c.ctx - key0 : 0;
  g.n_new = min(c.ctx + c.Mb - key0, KT) - g.rr0;    // >= 1
  g.first_new = key0 + g.rr0 - c.ctx;
  return g;
}
// Where key tile t of pair (b, h) lives: the TMA coordinates (z, y) of its first key and the
// cache row of that key (rows of D elements).  Contiguous cache: z = b Hkv + h, y = t KT, row =
// z cap + y.  Paged cache (one pool per kv head, [Hkv][num_pages][KT][D]): page = block_table[b][t]
// (an id outside the pool is flagged and page 0 is used instead), z = h num_pages + page, y = 0,
// row = z KT; pages allocated in order then give each head one unbroken run, as the contiguous
// cache does.
struct KvTile {
  int z, y;
  size_t row;
};
__device__ __forceinline__ KvTile kv_tile_page(const AttnArgs& a, int page, int h) {
  if (page < 0 || page >= a.num_pages) {
    set_status(a.status, 0x2F2u);
    page = 0;
  }
  const int z = h * a.num_pages + page;
  return KvTile{z, 0, (size_t)z * KT};
}
__device__ __forceinline__ KvTile kv_tile(const AttnArgs& a, int b, int h, int t) {
  if (a.block_table == nullptr) {
    const int z = b * a.Hkv + h;
    return KvTile{z, t * KT, (size_t)z * a.cap + (size_t)t * KT};
  }
  return kv_tile_page(a, a.block_table[(size_t)b * a.max_pages + t], h);
}

// NT threads load the new rows of head h from `src` (row stride ldkv) into registers:
// 16-byte chunk t + NT k of the n_new x 16 chunks (the block has at most 64 rows).
template <int NT>
__device__ __forceinline__ void tail_load(uint4 (&v)[1024 / NT], const uint16_t* src, const Cursor& c,
                                          const TailRows& g, int ldkv, int t) {
#pragma unroll
  for (int k = 0; k < 1024 / NT; ++k) {
    const int idx = t + NT * k, j = idx >> 4, ch = idx & 15;
    v[k] = make_uint4(0, 0, 0, 0);
    if (j < g.n_new)
      v[k] = *reinterpret_cast<const uint4*>(src + (size_t)(c.r0 + g.first_new + j) * ldkv + (size_t)c.h * D + ch * 8);
  }
}
// ... and store them into the landed stage and into the cache rows of pair bh.  Only the CTA
// owning the tile loads those cache rows, and its load has landed.  With `zero_rest` the stage
// rows past the new block are zeroed: whatever the cache holds there would meet P = 0 in P . V
// (K needs no zeros: masked scores are replaced, not multiplied).
template <int NT>
__device__ __forceinline__ void tail_store(const uint4 (&v)[1024 / NT], uint8_t* stage, uint16_t* cache,
                                           const TailRows& g, size_t row0, int t, bool zero_rest) {
#pragma unroll
  for (int k = 0; k < 1024 / NT; ++k) {
    const int idx = t + NT * k, j = idx >> 4, ch = idx & 15;
    if (j < g.n_new) {
      const int rr = g.rr0 + j;
      *reinterpret_cast<uint4*>(stage + (ch >> 3) * KV_HALF + sw128_off(rr, (ch & 7) * 8)) = v[k];
      *reinterpret_cast<uint4*>(cache + (row0 + rr) * D + ch * 8) = v[k];
    }
  }
  if (zero_rest)
    for (int idx = (g.rr0 + g.n_new) * 16 + t; idx < KT * 16; idx += NT) {
      const int rr = idx >> 4, ch = idx & 15;
      *reinterpret_cast<uint4*>(stage + (ch >> 3) * KV_HALF + sw128_off(rr, (ch & 7) * 8)) = make_uint4(0, 0, 0, 0);
    }
}

__global__ void __launch_bounds__(THREADS, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int* g_pfx = a.pfx + (size_t)blockIdx.x * (a.B + 1);
  const Meta meta{g_pfx, a.ctx_len, a.cu_rows};
  int* s_pfx = reinterpret_cast<int*>(smem + OFF_V);
  int* s_ctx = s_pfx + (a.B + 1);
  int* s_cu = s_ctx + a.B;
  const Meta smeta{s_pfx, s_ctx, s_cu};
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* k_full = bars;                 // [ST_K] K tile ready (tiles with new keys: after the patch)
  uint64_t* k_empty = k_full + ST_K;       // [ST_K] QK^T done with the K stage
  uint64_t* k_land = k_empty + ST_K;       // [ST_K] load landed of a tile that gets new keys
  uint64_t* v_full = k_land + ST_K;        // [ST_V]
  uint64_t* v_empty = v_full + ST_V;       // [ST_V] PV done with the V stage
  uint64_t* v_land = v_empty + ST_V;       // [ST_V]
  uint64_t* s_full = v_land + ST_V;        // [2]    S in TMEM
  uint64_t* s_empty = s_full + 2;          // [2]    softmax has read S
  uint64_t* p_full = s_empty + 2;          //        P in smem, O rescaled
  uint64_t* pv_done = p_full + 1;          //        PV finished (P free, O current)
  uint64_t* o_empty = pv_done + 1;         // [2]    epilogue has read the O buffer
  uint64_t* q_full = o_empty + 2;          // [QB]   Q of a pair staged
  uint64_t* q_empty = q_full + QB;         // [QB]   last QK^T of a pair done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + N_BARS);
  unsigned* last_flag = reinterpret_cast<unsigned*>(smem + OFF_FLAG);
  long long* s_range = reinterpret_cast<long long*>(bars + N_BARS + 1);   // this CTA's [ub, ue), units
  Cursor* s_cur = reinterpret_cast<Cursor*>(smem + OFF_FLAG + 8);         // the cursor at ub

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int B = a.B, Hkv = a.Hkv, G = a.G;
  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int s = 0; s < ST_K; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&k_land[s], 1);
    }
    for (int s = 0; s < ST_V; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&v_land[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 128);
      mbar_init(&o_empty[i], 128);
    }
    for (int i = 0; i < QB; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(tmem_slot, TMEM_COLS);
  // the shared-memory and TMEM setup above overlaps the previous kernel; global memory only below
  pdl_wait();
  pdl_trigger();

  // ---- per-sequence metadata: one parallel load, then a warp-0 scan of the tile counts (kept
  // in shared memory for the searches below and copied to this CTA's prefix slice for merges)
  for (int b = tid; b <= B; b += THREADS) {
    s_cu[b] = a.cu_rows[b];
    if (b < B) s_ctx[b] = a.ctx_len[b];
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    bool bad = false;
    for (int base = 0; base < B; base += 32) {
      const int b = base + lane;
      int units = 0;
      if (b < B) {
        const int ctx = s_ctx[b];
        const int mb = s_cu[b + 1] - s_cu[b];
        const int cap_keys = a.block_table ? a.max_pages * KT : a.cap;
        bad |= (mb <= 0 || mb > a.max_rows || ctx < 0 || ctx + mb > cap_keys || G * mb > QR);
        units = (mb > 0 && ctx >= 0) ? (ctx + mb + KT - 1) / KT * Hkv : 0;
      }
      int incl = units;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (b < B) s_pfx[b] = g_pfx[b] = carry + incl - units;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      s_pfx[B] = g_pfx[B] = bad ? 0 : carry;   // nothing to do when the ragged arrays are invalid
      if (bad && blockIdx.x == 0) set_status(a.status, 0x2F1u);
    }
    __syncwarp();
    if (lane == 0) {
      const long long U = s_pfx[B];
      const Part q{U, WT * U + (long long)a.pair_cost * B * Hkv, B * Hkv, (int)gridDim.x, Hkv, a.pair_cost};
      s_range[0] = range_start(q, smeta, blockIdx.x);
      s_range[1] = range_start(q, smeta, blockIdx.x + 1);
      s_range[2] = U;
      if (s_range[1] > s_range[0]) *s_cur = cur_at(smeta, B, s_range[0]);
    }
  }
  // the V ring's metadata copy is dead from here: order its generic accesses before the TMA writes
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long total = s_range[2];
  const Part part{total, WT * total + (long long)a.pair_cost * B * Hkv, B * Hkv, (int)gridDim.x, Hkv, a.pair_cost};
  const long long ub = s_range[0], ue = s_range[1];
  const long long n_units = ue - ub;

  if (warp == 4 || warp == 6) {
    // ------------------------------------------------------------ TMA producers: K and V
    if (lane == 0 && n_units > 0) {
      const bool is_k = warp == 4;
      const int nst = is_k ? ST_K : ST_V;
      const CUtensorMap* tm = is_k ? &tmK : &tmV;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint64_t* land = is_k ? k_land : v_land;
      uint8_t* ring = smem + (is_k ? OFF_K : OFF_V);
      const uint64_t pol = l2_policy_evict_first();
      Cursor c = *s_cur;
      // paged cache: the block-table entries are read PF units ahead of the loads that use them
      // (a second cursor), so a page lookup's latency never sits in front of a TMA issue
      constexpr int PF = 4;
      int pq[PF] = {0, 0, 0, 0};
      Cursor ca = c;
      const bool paged = a.block_table != nullptr;
      if (paged) {
#pragma unroll
        for (int j = 0; j < PF; ++j)
          if (j < n_units) {
            if (j > 0) cur_next(ca, meta, B, Hkv);
            pq[j] = a.block_table[(size_t)ca.b * a.max_pages + ca.t];
          }
      }
      for (long long i = 0; i < n_units; ++i, cur_next(c, meta, B, Hkv)) {
        const int s = (int)(i % nst);
        const int key0 = c.t * KT;
        const int page = pq[0];
        if (paged) {
#pragma unroll
          for (int j = 0; j + 1 < PF; ++j) pq[j] = pq[j + 1];
          if (i + PF < n_units) {
            cur_next(ca, meta, B, Hkv);
            pq[PF - 1] = a.block_table[(size_t)ca.b * a.max_pages + ca.t];
          }
        }
        if (i >= nst &&
            !mbar_wait(&empty[s], (uint32_t)(((i / nst) - 1) & 1), a.status, is_k ? 0x211u : 0x212u))
          break;
        uint64_t* bar = (key0 + KT > c.ctx) ? &land[s] : &full[s];
        uint8_t* st = ring + s * KV_TILE;
        const KvTile kt = paged ? kv_tile_page(a, page, c.h) : kv_tile(a, c.b, c.h, c.t);
        mbar_arrive_expect_tx(bar, KV_TILE);
        tma_load_3d_hint(st, tm, bar, 0, kt.y, kt.z, pol);
        tma_load_3d_hint(st + KV_HALF, tm, bar, 64, kt.y, kt.z, pol);
      }
    }
    __syncwarp();
  } else if (warp == 7) {
    // ------------------------------------------------------------ Q staging + new K rows
    bool ok = true;
    int piece = -1;
    int n_land_k[ST_K] = {};
    Cursor c = n_units > 0 ? *s_cur : Cursor{};
    for (long long i = 0; i < n_units && ok; ++i, cur_next(c, meta, B, Hkv)) {
      if (c.u == ub || c.t == 0) {
        // a new pair: its Q rows (row j = token row j / G, head j % G), zero-padded to 64,
        // loaded into registers first, stored once the last QK^T of the pair QB back is done
        ++piece;
        const int qb = piece % QB;
        const int R = G * c.Mb, ch = lane & 15;
        uint4 v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int j = 2 * k + (lane >> 4);
          v[k] = make_uint4(0, 0, 0, 0);
          if (j < R) {
            const int tr = j / G, g = j - tr * G;
            v[k] = *reinterpret_cast<const uint4*>(a.Q + (size_t)(c.r0 + tr) * a.ldq + (size_t)(c.h * G + g) * D + ch * 8);
          }
        }
        if (piece >= QB) ok = mbar_wait(&q_empty[qb], (uint32_t)((piece / QB - 1) & 1), a.status, 0x210u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        uint8_t* qd = smem + OFF_Q + qb * 2 * Q_HALF;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int j = 2 * k + (lane >> 4);
          *reinterpret_cast<uint4*>(qd + (ch >> 3) * Q_HALF + sw128_off(j, (ch & 7) * 8)) = v[k];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full[qb]);
      }
      if (c.t * KT + KT > c.ctx) {
        const int sk = (int)(i % ST_K);
        const TailRows g = tail_rows(c);
        uint4 v[32];
        tail_load<32>(v, a.Knew, c, g, a.ldkv, lane);
        ok = mbar_wait(&k_land[sk], (uint32_t)(n_land_k[sk]++ & 1), a.status, 0x213u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tail_store<32>(v, smem + OFF_K + sk * KV_TILE, a.Kc, g, kv_tile(a, c.b, c.h, c.t).row, lane, false);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&k_full[sk]);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer (event driven)
    if (lane == 0 && n_units > 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(QR, KT);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(QR, D) | (1u << 16);   // B (V) MN-major
      Cursor cs = *s_cur, cp = cs;
      long long ns = 0, np = 0;          // next QK^T, next PV
      int piece_s = -1, piece_p = -1;
      uint32_t spin = 0;
      uint64_t t0 = 0;
      while (np < n_units) {
        bool did = false;
        if (ns < n_units) {
          const bool first = (cs.u == ub || cs.t == 0);
          const bool last = (cs.u + 1 == ue) || (cs.t + 1 == cs.nt);
          const int pc = first ? piece_s + 1 : piece_s;
          const int qb = pc % QB, s = (int)(ns % ST_K);
          if ((!first || mbar_test(&q_full[qb], (uint32_t)((pc / QB) & 1))) &&
              mbar_test(&k_full[s], (uint32_t)((ns / ST_K) & 1)) &&
              (ns < 2 || mbar_test(&s_empty[ns & 1], (uint32_t)(((ns >> 1) - 1) & 1)))) {
            piece_s = pc;
            tc_fence_after();
            const uint32_t k_addr = smem_u32(smem + OFF_K + s * KV_TILE);
            const uint32_t q_addr = smem_u32(smem + OFF_Q + qb * 2 * Q_HALF);
            const uint32_t d_s = tmem + (uint32_t)(ns & 1) * KT;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t qa = q_addr + (kk >> 2) * Q_HALF + (kk & 3) * 32;
              const uint32_t ka = k_addr + (kk >> 2) * KV_HALF + (kk & 3) * 32;
              umma_bf16(d_s, umma_desc_sw128(qa), umma_desc_sw128(ka), idesc_s, kk > 0 ? 1u : 0u);
            }
            umma_commit(&k_empty[s]);
            umma_commit(&s_full[ns & 1]);
            if (last) umma_commit(&q_empty[qb]);
            ++ns;
            cur_next(cs, meta, B, Hkv);
            did = true;
          }
        }
        if (np < ns) {
          const bool first = (cp.u == ub || cp.t == 0);
          const int pc = first ? piece_p + 1 : piece_p;
          const int ob = pc & 1, s = (int)(np % ST_V);
          if (mbar_test(p_full, (uint32_t)(np & 1)) &&
              mbar_test(&v_full[s], (uint32_t)((np / ST_V) & 1)) &&
              (!first || pc < 2 || mbar_test(&o_empty[ob], (uint32_t)(((pc >> 1) - 1) & 1)))) {
            piece_p = pc;
            tc_fence_after();
            const uint32_t v_addr = smem_u32(smem + OFF_V + s * KV_TILE);
            const uint32_t p_addr = smem_u32(smem + OFF_P);
            const uint32_t t_o = tmem + 2 * KT + (uint32_t)ob * D;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t pa = p_addr + (kk >> 2) * Q_HALF + (kk & 3) * 32;
              const uint32_t va = v_addr + kk * 16 * 128;                     // 16 keys per step
              umma_bf16(t_o, umma_desc_sw128(pa), umma_desc_sw128_mn(va, KV_HALF), idesc_pv,
                        (!first || kk > 0) ? 1u : 0u);
            }
            umma_commit(&v_empty[s]);
            umma_commit(pv_done);
            ++np;
            cur_next(cp, meta, B, Hkv);
            did = true;
          }
        }
        if (did) {
          spin = 0;
        } else {
          if (spin == 0) t0 = globaltimer();
          if ((++spin & 1023u) == 0 && globaltimer() - t0 > SPEC_WAIT_NS) {
            set_status(a.status, 0x220u);
            break;
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue warps
    // Query row 16 q + (lane % 16) of warp q sits in TMEM lane 32 q + lane % 16; the two
    // half-warps share it, lanes 0-15 taking keys (and output dims) 0-63, lanes 16-31 keys
    // 64-127.  After a timed-out wait a thread stops waiting but keeps the same control
    // flow, so the named barriers below stay matched.
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    const int row = warp * 16 + (lane & 15);
    const int half = lane >> 4;
    const float scale = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int piece = -1;
    int n_land_v[ST_V] = {};
    Cursor c = n_units > 0 ? *s_cur : Cursor{};
    for (long long i = 0; i < n_units; ++i, cur_next(c, meta, B, Hkv)) {
      const long long u = c.u;
      const int R = G * c.Mb;
      const bool first = (u == ub || c.t == 0);
      const bool last = (u + 1 == ue) || (c.t + 1 == c.nt);
      if (first) {
        ++piece;
        m_run = -INFINITY;
        l_run = 0.f;
      }
      const int ob = piece & 1;
      const uint32_t t_o = tmem + 2 * KT + (uint32_t)ob * D + lane_off;
      const int key0 = c.t * KT;
      const bool tail = key0 + KT > c.ctx;
      // a tile with new keys: their V rows are fetched now and patched in before this tile's PV
      TailRows g{};
      uint4 vnew[8];
      if (tail) {
        g = tail_rows(c);
        tail_load<128>(vnew, a.Vnew, c, g, a.ldkv, tid);
      }
      // key k of this thread's half is visible to the row iff k <= lim (rows past the group
      // clamp to the last one)
      const int lim = c.ctx + min(row / G, c.Mb - 1) - key0 - half * 64;
      ok = ok && mbar_wait(&s_full[i & 1], (uint32_t)((i >> 1) & 1), a.status, 0x231u);
      tc_fence_after();
      float sv[64];
      tmem_ld_split64(tmem + (uint32_t)(i & 1) * KT + lane_off, sv);
      tc_fence_before();
      mbar_arrive(&s_empty[i & 1]);
      // scaled logits and their maximum (8 independent chains)
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
      for (int k = 0; k < 64; ++k) {
        float v = sv[k] * scale;
        if (tail && k > lim) v = -INFINITY;
        sv[k] = v;
        mx8[k & 7] = fmaxf(mx8[k & 7], v);
      }
      float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      // the running max only moves when the tile max exceeds it by more than 2^8: P <= 256
      // stays representable, and O, l keep using one common max, so the result is unchanged
      const float m_new = (mx > m_run + 8.f) ? mx : m_run;
      const bool grew = m_new != m_run;
      const float base = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ex2(m_run - base);
      float sm8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) sm8[e] = 0.f;
#pragma unroll
      for (int k = 0; k < 64; ++k) {
        sv[k] = ex2(sv[k] - base);
        sm8[k & 7] += sv[k];
      }
      float sm = ((sm8[0] + sm8[1]) + (sm8[2] + sm8[3])) + ((sm8[4] + sm8[5]) + (sm8[6] + sm8[7]));
      sm += __shfl_xor_sync(0xffffffffu, sm, 16);
      l_run = l_run * alpha + sm;
      m_run = m_new;
      // P was last read by PV(i - 1), which also has to be in O before O is rescaled
      if (i >= 1) ok = ok && mbar_wait(pv_done, (uint32_t)((i - 1) & 1), a.status, 0x232u);
      {
        uint8_t* prow = smem + OFF_P + half * Q_HALF;
#pragma unroll
        for (int k = 0; k < 64; k += 8) {
          const uint4 wv = make_uint4(pack_bf16x2(sv[k], sv[k + 1]), pack_bf16x2(sv[k + 2], sv[k + 3]),
                                      pack_bf16x2(sv[k + 4], sv[k + 5]), pack_bf16x2(sv[k + 6], sv[k + 7]));
          *reinterpret_cast<uint4*>(prow + sw128_off(row, k)) = wv;
        }
      }
      if (!first && __any_sync(0xffffffffu, grew)) {
        tc_fence_after();
        float ov[64];
        tmem_ld_split64(t_o, ov);
#pragma unroll
        for (int cc = 0; cc < 64; cc += 16) {
          float o16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) o16[e] = ov[cc + e] * alpha;
          tmem_st_split16(t_o + cc, o16);
        }
        tmem_st_wait();
      }
      if (tail) {
        const int sv_ = (int)(i % ST_V);
        ok = ok && mbar_wait(&v_land[sv_], (uint32_t)(n_land_v[sv_]++ & 1), a.status, 0x214u);
        tail_store<128>(vnew, smem + OFF_V + sv_ * KV_TILE, a.Vc, g, kv_tile(a, c.b, c.h, c.t).row, tid, true);
        fence_proxy_async_smem();
        bar_compute();
        if (tid == 0) mbar_arrive(&v_full[sv_]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
      if (!last) continue;

      // ---- piece epilogue: this thread's 64 output dims of the row once the tile's PV is done
      ok = ok && mbar_wait(pv_done, (uint32_t)(i & 1), a.status, 0x233u);
      tc_fence_after();
      float ov[64];
      tmem_ld_split64(t_o, ov);
      tc_fence_before();
      mbar_arrive(&o_empty[ob]);
      const int bh = c.b * Hkv + c.h;
      const long long pair0 = u - c.t;
      const long long pair_last = pair0 + c.nt - 1;
      const bool complete = (pair0 >= ub) && (u == pair_last);
      if (row < R) {
        if (complete) {
          const int tr = row / G, g = row - tr * G;
          store_half_bf16(a.O + (size_t)(c.r0 + tr) * a.ldo + (size_t)(c.h * G + g) * D + half * 64, ov, 1.f / l_run);
        } else {
          // slot 0: the piece that opens this CTA's range; slot 1: the piece that closes it
          const int slot = (pair0 < ub) ? 0 : 1;
          float* pb = a.partial + ((size_t)blockIdx.x * 2 + slot) * (QR * (D + 2));
#pragma unroll
          for (int d = 0; d < 64; d += 4)
            __stcg(reinterpret_cast<float4*>(pb + row * D + half * 64 + d),
                   make_float4(ov[d], ov[d + 1], ov[d + 2], ov[d + 3]));
          if (half == 0) __stcg(reinterpret_cast<float2*>(pb + QR * D + row * 2), make_float2(m_run, l_run));
        }
      }
      if (complete) continue;
      // ---- split pair: count this piece's tiles; the last arrival merges in CTA order
      __threadfence();
      bar_compute();
      if (tid == 0) {
        const long long piece_first = pair0 > ub ? pair0 : ub;
        const unsigned add = (unsigned)(u - piece_first + 1);
        const unsigned prev = atomicAdd(&a.counters[bh], add);
        *last_flag = (prev + add == (unsigned)c.nt) ? 1u : 0u;
      }
      bar_compute();
      const bool merge = *last_flag != 0u;
      bar_compute();
      if (!merge) continue;
      __threadfence();
      const int p_id = c.b * Hkv + c.h;
      const int c_lo = cta_of(part, pair0, p_id);
      const int c_hi = cta_of(part, pair_last, p_id);
      // one pass over the contributors in CTA order (each one's (m, l) and O half-row loaded
      // together), rescaling the running sums to the running maximum.  The first contributor
      // left its piece in slot 1 (the pair starts inside its range), the others in slot 0;
      // a CTA between them with an empty range contributed nothing.
      if (row < R) {
        float M = -INFINITY, L = 0.f;
        float acc[64];
#pragma unroll
        for (int d = 0; d < 64; ++d) acc[d] = 0.f;
        long long next_start = c_hi - c_lo >= 2 ? range_start(part, meta, c_lo + 1) : 0;
        for (int c2 = c_lo; c2 <= c_hi; ++c2) {
          if (c2 > c_lo && c2 < c_hi) {
            const long long st = next_start;
            next_start = range_start(part, meta, c2 + 1);
            if (next_start == st) continue;
          }
          const int sl = c2 == c_lo ? 1 : 0;
          const float* pk = a.partial + ((size_t)c2 * 2 + sl) * (QR * (D + 2));
          const float2 ml = __ldcg(reinterpret_cast<const float2*>(pk + QR * D + row * 2));
          float4 v[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] = __ldcg(reinterpret_cast<const float4*>(pk + row * D + half * 64 + q * 4));
          const float mn = fmaxf(M, ml.x);
          if (mn == -INFINITY) continue;                       // nothing visible in either yet
          const float fo = ex2(M - mn), fc = ex2(ml.x - mn);  // 2^-inf = 0
          L = L * fo + ml.y * fc;
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            acc[4 * q] = acc[4 * q] * fo + v[q].x * fc;
            acc[4 * q + 1] = acc[4 * q + 1] * fo + v[q].y * fc;
            acc[4 * q + 2] = acc[4 * q + 2] * fo + v[q].z * fc;
            acc[4 * q + 3] = acc[4 * q + 3] * fo + v[q].w * fc;
          }
          M = mn;
        }
        const int tr = row / G, g = row - tr * G;
        store_half_bf16(a.O + (size_t)(c.r0 + tr) * a.ldo + (size_t)(c.h * G + g) * D + half * 64, acc, 1.f / L);
      }
      if (tid == 0) a.counters[bh] = 0u;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

int attention_tc_key_tile() { return KT; }
int attention_tc_max_batch() { return MAX_B; }
int attention_tc_rows(int G, int max_rows) { return G * max_rows <= QR ? QR : -1; }

cudaError_t launch_attention_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, int grid,
                                cudaStream_t s) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  cudaError_t e = launch_k(attention_tc_kernel, dim3(grid), dim3(THREADS), SMEM, s, tk, tv, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace spec
