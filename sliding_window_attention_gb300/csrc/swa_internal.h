// Internal interface between the C-ABI translation unit and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

namespace swa {

// Problem geometry shared by every kernel.  There are Lq query rows and L
// key rows (Lq <= L); the queries are the last Lq positions of the key
// sequence, so query row i sits at key position i + off with off = L - Lq
// (the pages' diag_off; 0 for self-attention).
struct Geom {
  int B, Hq, Hkv, L, D, W, G;  // L = key rows; G = Hq / Hkv; W = 0: no window
  int Lq, off;                 // query rows, L - Lq
  int causal;                  // 1: keys after the query's position are masked
  float scale;                 // softmax scale applied to q . k
  // Shared-prefix plan (Rc > 0): one causal self-attention pass over
  // [prompt (P rows); chosen response (Rc rows); rejected response (the
  // rest)] in which rejected rows do not see chosen keys and the window is
  // measured on logical positions, the rejected response restarting at P.
  // Rc == 0: no plan.  With a plan, Lq == L, off == 0, causal == 1 and
  // P + Rc < L.
  int P, Rc;
  // Attention sinks: one logit per query head ([Hq] fp32, device memory),
  // an extra term of every row's softmax normaliser that carries no value,
  // or nullptr for none.  Not combined with a plan.
  const float* sinks;
};

// Folds a sink logit c (natural-log units) into a row's final softmax
// normaliser.  m2 is the row's reference maximum in log2 units and l its sum
// of 2^(score - m2) terms; O is the accumulated P V for those terms.  With
// mf = max(m2, c log2 e):
//   l' = l 2^(m2 - mf) + 2^(c log2 e - mf),   lse = (mf + log2 l') ln 2,
// and the row's output is O times the returned factor 2^(m2 - mf) / l'
// (1 / l when the sink is -inf).  m2 = -inf (a row without keys) gives a
// factor of 0 and lse = c.
__device__ __forceinline__ float sink_finish(float c, float m2, float l, float* lse) {
  const float c2 = c * 1.4426950408889634f;
  const float mf = fmaxf(m2, c2);
  const float a = exp2f(m2 - mf);
  const float lf = fmaf(l, a, exp2f(c2 - mf));
  *lse = (mf + log2f(lf)) * 0.6931471805599453f;
  return a / lf;
}

// The band of query row i is the interval of keys [band_key_lo, band_key_hi]
// ("Lab 028 lab detail: Off NVIDIA, you fix the platform yourself", "Plan
// for the build" step 4 and "What I changed, in plain terms" items 3-4):
//   causal:      j <= a and (W == 0 or a - j < W),  a = i + off
//   non-causal:  W == 0 or |a - j| < W
// Both ends are non-decreasing in i, and the rows that see key j form the
// interval [band_q_lo, band_q_hi] (empty when lo > hi).
//
// Under a shared-prefix plan ("Training -- design (ORPO, flash-CCE head,
// prefix sharing, segmented backward)", section 5.4: causal AND NOT
// rejected -> chosen, window on logical positions) a row or a key sees up to
// two intervals, `part` 0 and 1, which are disjoint:
//   rejected row i:  part 0 = prompt keys [i - Rc - W + 1, P - 1],
//                    part 1 = rejected keys [max(P + Rc, i - W + 1), i];
//   other rows:      part 0 = the plain causal window, part 1 empty;
//   prompt key j:    part 0 = prompt and chosen rows [j, min(P + Rc - 1, j + W - 1)],
//                    part 1 = rejected rows [P + Rc, j + Rc + W - 1];
//   other keys:      part 0 = the rows of their own response within the
//                    window, part 1 empty.
// (W == 0 drops the window bounds.)  Without a plan part 0 is the band above
// and part 1 is empty.  An empty interval has lo > hi.
__host__ __device__ __forceinline__ int band_key_lo(const Geom& g, int i, int part = 0) {
  if (g.Rc > 0 && i >= g.P + g.Rc) {
    const int lo = part ? i - g.W + 1 : i - g.Rc - g.W + 1;
    const int floor_ = part ? g.P + g.Rc : 0;
    return (g.W > 0 && lo > floor_) ? lo : floor_;
  }
  if (part) return g.L;
  const int lo = i + g.off - g.W + 1;
  return (g.W > 0 && lo > 0) ? lo : 0;
}
__host__ __device__ __forceinline__ int band_key_hi(const Geom& g, int i, int part = 0) {
  if (g.Rc > 0 && i >= g.P + g.Rc) return part ? i : g.P - 1;
  if (part) return -1;
  const int a = i + g.off;
  const int hi = g.causal ? a : (g.W > 0 ? a + g.W - 1 : g.L - 1);
  return hi < g.L - 1 ? hi : g.L - 1;
}
__host__ __device__ __forceinline__ int band_q_lo(const Geom& g, int j, int part = 0) {
  if (part) return (g.Rc > 0 && j < g.P) ? g.P + g.Rc : g.Lq;
  if (!g.causal && g.W == 0) return 0;
  const int lo = (g.causal ? j : j - g.W + 1) - g.off;
  return lo > 0 ? lo : 0;
}
__host__ __device__ __forceinline__ int band_q_hi(const Geom& g, int j, int part = 0) {
  if (g.Rc > 0) {
    if (part) {
      if (j >= g.P) return -1;
      const int hi = g.W > 0 ? j + g.Rc + g.W - 1 : g.L - 1;
      return hi < g.L - 1 ? hi : g.L - 1;
    }
    const int seg_end = j < g.P + g.Rc ? g.P + g.Rc - 1 : g.L - 1;  // rows of the key's own block
    const int hi = g.W > 0 ? j + g.W - 1 : g.L - 1;
    return hi < seg_end ? hi : seg_end;
  }
  if (part) return -1;
  if (g.W == 0) return g.Lq - 1;
  const int hi = j + g.W - 1 - g.off;
  return hi < g.Lq - 1 ? hi : g.Lq - 1;
}

// Visible columns of one row (or key) inside a tile starting at c0: the two
// intervals [x, y] and [z, w] in tile-local coordinates.
__host__ __device__ __forceinline__ int4 row_vis(const Geom& g, int i, int c0) {
  return make_int4(band_key_lo(g, i, 0) - c0, band_key_hi(g, i, 0) - c0, band_key_lo(g, i, 1) - c0,
                   band_key_hi(g, i, 1) - c0);
}
__host__ __device__ __forceinline__ int4 key_vis(const Geom& g, int j, int c0) {
  return make_int4(band_q_lo(g, j, 0) - c0, band_q_hi(g, j, 0) - c0, band_q_lo(g, j, 1) - c0,
                   band_q_hi(g, j, 1) - c0);
}
// The same intervals seen from a column offset d further into the tile.
__host__ __device__ __forceinline__ int4 vshift(const int4& v, int d) {
  return make_int4(v.x - d, v.y - d, v.z - d, v.w - d);
}
// The visible columns of one row in a tile of T columns, in tile-local
// coordinates: when only one of the two intervals meets the tile it moves to
// the first slot (the second is emptied), and *both says whether both meet
// it (under a shared-prefix plan only where the gap between them falls inside
// the tile).  A row that sees nothing of the tile gets an empty first slot.
__host__ __device__ __forceinline__ int4 vis_in_tile(const int4& v, int T, bool* both) {
  const bool a = v.x <= v.y && v.y >= 0 && v.x < T;
  const bool b = v.z <= v.w && v.w >= 0 && v.z < T;
  *both = a && b;
  if (a && b) return v;
  if (b) return make_int4(v.z, v.w, 1, 0);
  if (a) return make_int4(v.x, v.y, 1, 0);
  return make_int4(1, 0, 1, 0);
}
// Column c of a masked tile is visible: in [v.x, v.y], or (TWO: a plan is
// active) in [v.z, v.w].
template <bool TWO>
__host__ __device__ __forceinline__ bool vis(int c, const int4& v) {
  return (c >= v.x && c <= v.y) || (TWO && c >= v.z && c <= v.w);
}

// The tiles one CTA visits: those that meet the part-0 hull, then those that
// meet the part-1 hull and not the part-0 one (a tile that meets both is
// visited once, masked with both intervals).
struct TileSteps {
  int lo0, n0, lo1, n1;
  __host__ __device__ int count() const { return n0 + n1; }
  __host__ __device__ int tile(int n) const { return n < n0 ? lo0 + n : lo1 + (n - n0); }
};
__host__ __device__ __forceinline__ TileSteps make_steps(int lo0, int hi0, int lo1, int hi1, int T) {
  TileSteps s;
  s.lo0 = lo0 <= hi0 ? lo0 / T : 0;
  s.n0 = lo0 <= hi0 ? hi0 / T - lo0 / T + 1 : 0;
  int a = lo1 / T, z = hi1 / T;
  if (s.n0 > 0 && a <= s.lo0 + s.n0 - 1) a = s.lo0 + s.n0;  // tiles already in part 0
  s.lo1 = a;
  s.n1 = (lo1 <= hi1 && a <= z) ? z - a + 1 : 0;
  return s;
}
// Key tiles (of T keys) that rows [r0, r1] see.
__host__ __device__ __forceinline__ TileSteps row_steps(const Geom& g, int r0, int r1, int T) {
  if (g.Rc == 0) return make_steps(band_key_lo(g, r0), band_key_hi(g, r1), 1, 0, T);
  const int R = g.P + g.Rc;  // first rejected row
  int lo0 = g.L, hi0 = -1;
  if (r0 < R) {  // rows of the prompt and the chosen response: the plain causal window
    lo0 = band_key_lo(g, r0, 0);
    hi0 = band_key_hi(g, r1 < R ? r1 : R - 1, 0);
  }
  int lo1 = g.L, hi1 = -1;
  if (r1 >= R) {  // rejected rows: prompt keys (part 0, shrinking) and rejected keys (part 1)
    const int a = r0 > R ? r0 : R;
    const int l = band_key_lo(g, a, 0), h = band_key_hi(g, a, 0);
    if (l <= h) {
      lo0 = l < lo0 ? l : lo0;
      hi0 = h > hi0 ? h : hi0;
    }
    lo1 = band_key_lo(g, a, 1);
    hi1 = r1;
  }
  return make_steps(lo0, hi0, lo1, hi1, T);
}
// Query tiles (of T rows) that see keys [j0, j1].
__host__ __device__ __forceinline__ TileSteps key_steps(const Geom& g, int j0, int j1, int T) {
  const int lo0 = band_q_lo(g, j0, 0), hi0 = band_q_hi(g, j1, 0);
  if (g.Rc == 0 || j0 >= g.P) return make_steps(lo0, hi0, 1, 0, T);
  const int jp = j1 < g.P - 1 ? j1 : g.P - 1;  // the tile's last prompt key
  return make_steps(lo0, hi0, g.P + g.Rc, band_q_hi(g, jp, 1), T);
}
// Every row of [r0, r1] sees every key of [c0, c1] (no mask needed).
__host__ __device__ __forceinline__ bool rows_tile_full(const Geom& g, int r0, int r1, int c0, int c1) {
  if (g.Rc == 0) return c0 >= band_key_lo(g, r1) && c1 <= band_key_hi(g, r0);
  const int R = g.P + g.Rc;
  if (r1 < R) return c0 >= band_key_lo(g, r1, 0) && c1 <= band_key_hi(g, r0, 0);
  if (r0 < R) return false;
  return (c0 >= band_key_lo(g, r1, 0) && c1 <= band_key_hi(g, r0, 0)) ||
         (c0 >= band_key_lo(g, r1, 1) && c1 <= band_key_hi(g, r0, 1));
}
// Every key of [j0, j1] is seen by every row of [c0, c1].
__host__ __device__ __forceinline__ bool keys_tile_full(const Geom& g, int j0, int j1, int c0, int c1) {
  if (c0 >= band_q_lo(g, j1, 0) && c1 <= band_q_hi(g, j0, 0)) return true;
  return g.Rc > 0 && j1 < g.P && c0 >= g.P + g.Rc && c1 <= band_q_hi(g, j0, 1);
}

// Device-side status codes latched into the per-device status word.
enum : int { kStatusOk = 0, kStatusTimeout = -11, kStatusFp16Range = -14, kStatusScratch = -15 };

// The head-dim-512 kernels hand tiles between the CTAs of a cluster through
// a static L2 scratch indexed by the SM id of the receiving CTA (192 SM ids).
// That needs at most one CTA of these kernels per SM and SM ids below 192.
// Each returns 0 when the current device meets that, 1 when it does not,
// and -1 when the CUDA queries fail.
int scratch_layout_fwd512();
int scratch_layout_bwd512();
// Head dim 256: the dK/dV clusters pass P^T through a static L2 scratch indexed
// by the dK CTA's SM id, under the same two conditions.
int scratch_layout_bwd256();

// ---- SIMT kernels (fp32 arithmetic on bf16 inputs; any D in {64..512}) ----
cudaError_t launch_fwd_simt(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            float* o, float* lse, cudaStream_t s);
cudaError_t launch_delta(const Geom& g, const float* o, const uint16_t* dO, float* delta, cudaStream_t s);
cudaError_t launch_bwd_dkdv_simt(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 const uint16_t* dO, const float* lse, const float* delta, float* dk,
                                 float* dv, cudaStream_t s);
cudaError_t launch_bwd_dq_simt(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const uint16_t* dO, const float* lse, const float* delta, float* dq,
                               cudaStream_t s);

// ---- tensor-core path (tcgen05 + TMA + TMEM), fp16 operand copies ----
// bf16 -> fp16 copies of up to four tensors (n[i] elements, multiples of 8);
// latches kStatusFp16Range in *status if a finite input overflows fp16; sets
// *zero_word to 0 when it is not null (the work counter of a persistent
// launch that follows on the stream).
cudaError_t launch_convert_f16(const uint16_t* const* src, uint16_t* const* dst, const size_t* n, int count,
                               int* status, cudaStream_t s, int* zero_word = nullptr);
// One CTA whose bounded wait on a barrier nothing completes runs out after
// limit_cycles and latches kStatusTimeout in *status.
cudaError_t launch_selftest_timeout(int* status, long long limit_cycles, cudaStream_t s);
bool fwd_tc_supported(int D);
// Decode-shaped forward (decode.cu): at most kDecodeMaxRows = G * Lq query
// rows per kv head, read as bf16 straight from q, k, v (no fp16 copies).
constexpr int kDecodeMaxRows = 16;
bool decode_supported(const Geom& g);
size_t decode_workspace_bytes(const Geom& g);  // fp32 chunk partials; 0 when one chunk suffices
cudaError_t launch_fwd_decode(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v, float* o,
                              float* lse, float* ws, int* status, cudaStream_t s);
// Head dim 512: persistent 4-CTA clusters (tc_fwd512.cu) that draw work
// items from *work, which must be zero when the launch starts.
cudaError_t launch_fwd_tc512(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v16, float* o,
                             float* lse, int* work, int* status, cudaStream_t s);
// Forward on the tensor cores: q and k are the caller's bf16 tensors (S = Q K^T
// runs on bf16 operands), v16 an fp16 copy of v (O += P V pairs it with fp16 P).
// work: a zeroed int in the workspace (used at head dim 512).
cudaError_t launch_fwd_tc(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v16, float* o,
                          float* lse, int* work, int* status, cudaStream_t s);

// 3-D fp16 tensor map over [heads, L, D] with a 64 x box_rows box and
// 128-byte swizzle (rows at or beyond L read as zero).
cudaError_t make_tmap_f16(CUtensorMap* m, const void* ptr, int D, int L, int heads, int box_rows);
// The same tensor as a 4-D map whose box (64, box_rows, nchunk, 1) loads
// nchunk 64-column chunks (consecutive [box_rows x 128 B] swizzled blocks)
// with one TMA instruction; coordinates (0, row, first chunk, head).
cudaError_t make_tmap_f16_chunks(CUtensorMap* m, const void* ptr, int D, int L, int heads, int box_rows,
                                 int nchunk);

// 3-D fp32 tensor map over an output [heads, L, D] for the D = 512 epilogues:
// 32 x 32 boxes (128-byte rows) with 128-byte swizzle; TMA stores clip rows
// at or beyond L.
cudaError_t make_tmap_f32_out(CUtensorMap* m, void* ptr, int D, int L, int heads);

bool bwd_tc_supported(int D);
// Padded row count of the backward's row-statistics array.
int bwd_stats_lpad(int L);

// The fp16 copy of dO is scaled by a power of two s, chosen from max |dO| so
// that the scaled maximum lies in [4, 8): tiny cotangents then keep their
// precision in fp16 (and large ones cannot overflow it) in dO and in
// dS = P (dP - Delta), which are linear in dO.  Delta is stored scaled by s
// too, and the dq, dk and dv epilogues multiply by 1/s, exactly.
// The backward's row-statistics block ends with a tail of
// kDScaleTailFloats floats at stats + dscale_offset(): [0] = s, [1] = 1/s,
// [2], [3] the work counters (int32) of the persistent head-dim-512 dK/dV and
// dQ passes, zeroed by the absmax pass, [4, 4 + kAbsmaxBlocks) per-block
// maxima of |dO| (bf16 bit patterns with the sign cleared, as uint32) written
// by the absmax pass.
constexpr int kAbsmaxBlocks = 304;
constexpr int kWorkCounterFloat = 2;
constexpr int kDScaleTailFloats = 4 + kAbsmaxBlocks;
__host__ __device__ __forceinline__ size_t dscale_offset(const Geom& g, int Lpad) {
  return 2 * (size_t)g.B * g.Hq * Lpad;
}
// max |dO| per block of the absmax pass into the stats tail, and the work
// counters zeroed (one launch).
cudaError_t launch_bwd_dscale(const Geom& g, int Lpad, const uint16_t* dO, float* stats, cudaStream_t s);
// Gradient of the attention sinks g.sinks into dsinks [Hq] (fp32), from the
// row statistics the backward prep wrote (run after the prep).
cudaError_t launch_sink_grad(const Geom& g, int Lpad, const float* stats, float* dsinks, cudaStream_t s);
// The backward's preparation in one pass (after launch_bwd_dscale): fp16
// copies of q, k, v and s * dO, and the row statistics, two planes of
// B * Hq * Lpad floats: stats[bh * Lpad + i] = lse_i * log2(e),
// stats[(B * Hq + bh) * Lpad + i] = s * (dO_i . o_i) (zero for i >= Lq); dO
// is read once here.  Also writes s and 1/s into the stats tail.
cudaError_t launch_bwd_prep(const Geom& g, int Lpad, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            const uint16_t* dO, const float* o, const float* lse, uint16_t* q16, uint16_t* k16,
                            uint16_t* v16, uint16_t* g16, float* stats, int* status, cudaStream_t s);
cudaError_t launch_bwd_dkdv_tc(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                               const uint16_t* g16, const float* stats, int Lpad, float* dk, float* dv,
                               int* status, cudaStream_t s);
// Head dim 512: thread-block-cluster kernels (tc_bwd512.cu).
// Head dim 512: the dK/dV and dQ passes on clusters of CTA pairs (tcgen05
// .cta_group::2).
cudaError_t launch_bwd_dkdv_tc512(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                                   const uint16_t* g16, const float* stats, int Lpad, float* dk, float* dv,
                                   int* status, cudaStream_t s);
// Both passes are persistent (as many clusters as fit at once, looping over
// work items from the stats tail's counters).  The dQ pass is launched with
// programmatic stream serialization: enqueued on the dK/dV pass's stream
// right after it, it starts on the SMs that pass leaves and completes after
// it.
cudaError_t launch_bwd_dq_tc512(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                                 const uint16_t* g16, const float* stats, int Lpad, float* dq, int* status,
                                 cudaStream_t s);
cudaError_t launch_bwd_dq_tc(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                             const uint16_t* g16, const float* stats, int Lpad, float* dq, int* status,
                             cudaStream_t s);

}  // namespace swa
