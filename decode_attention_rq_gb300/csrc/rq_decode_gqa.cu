// Grouped-query decode calls: the query heads that share a KV head score and
// weight one staged copy of its tiles.
//
// With Hq = qpk * H query heads, the per-head kernel (rq_decode_kernels.cuh)
// streams every KV tile once per query head.  Here a work unit is (row, head
// group, 128 tokens), a head group being QH = 2 or 4 consecutive query heads
// of one KV head, and the unit's tiles are read once for all of them:
//   * scoring: the K code operands are converted once; each head then runs its
//     own tensor-core products against its query images (kept in shared memory,
//     one set per head) and its own epilogue;
//   * softmax: a running maximum, denominator and offset sums per head;
//   * value products: the B operand of a value product has eight columns, of
//     which one head uses two (its weights' hi and lo f16 pieces).  Head h takes
//     columns 2h and 2h + 1, so one product over the V codes serves all QH
//     heads, and lane t's accumulators hold head t's sums.
// The query prep and merge kernels are the per-head ones: the prep writes one
// pack per query head, and the merge recomputes each head's contributing CTAs
// from the head-group split (DecodeArgs::qh).  With qpk = 8 the KV head's two
// head groups are neighbours in the work list, so their CTAs stream the same
// tiles at about the same time.
#include "rq_decode_kernels.cuh"

namespace rq {
namespace {

template <int D, int GS, int NRES, int QH>
struct GCfg {
  using L = Cfg<D, GS, NRES>;
  static constexpr int NITEM = L::NITEM, NIMG = L::NIMG;
  static constexpr int MINB = 2;   // CTAs per SM: the per-head state takes up to 128 registers a thread
  // Value-weight image of one (plane, group): one plane per B column (head h:
  // column 2h the hi pieces, 2h + 1 the lo pieces), each holding per value
  // product m (8) and lane t (4) the registers b0, b1 (8 B).  Planes 288 B apart
  // (8 banks), items 72 B further apart, as in the per-head images.
  static constexpr int NPL = 2 * QH;
  static constexpr int PLANE = 288;
  static constexpr int ITEM = NPL * PLANE + 72;
  // + a zero block for the lanes of unused columns; rounded so that the query operands start aligned
  static constexpr int WIMG = (NITEM * ITEM + 256 + 127) / 128 * 128;
  // Query operands in shared memory, per head: the pack header (32 words), then
  // nine lane images of IMS words: the eight of the pack and a zero image that
  // the lanes with zero B operands read.  IMS / 2 is odd, so the eight lanes'
  // 8-byte loads fall on distinct banks (the zero image's on others).
  static constexpr int IMS = NIMG + 2;
  static constexpr int QHEAD = kPackHeader + 9 * IMS;
  static constexpr int QIMG = (QH * QHEAD * 4 + 127) / 128 * 128;
  static constexpr int STAGE = L::STAGE;
  static constexpr int STAGES = (MINB * (3 * STAGE + WIMG + QIMG) + MINB * 8192 <= 224 * 1024) ? 3 : 2;
  static constexpr int SMEM = STAGES * STAGE + WIMG + QIMG;
  // heads whose scoring products run on one conversion of the codes (the rest
  // convert again: bounds the accumulators held at once)
  static constexpr int SC = (L::NACA + L::NACR <= 2) ? QH : 2;
  static_assert((IMS / 2) % 2 == 1, "lane images on distinct banks");
  static_assert(STAGE % 16 == 0 && WIMG % 16 == 0, "16-byte aligned regions");
  static_assert(QH % SC == 0, "scoring chunks");
};

template <int D, int GS, int NRES, bool PAGED, int QH>
__global__ void __launch_bounds__(kThreads, 2) decode_gqa_kernel(DecodeArgs a) {
  using C = Cfg<D, GS, NRES>;
  using G = GCfg<D, GS, NRES, QH>;
  constexpr int NG = C::NG, STAGES = G::STAGES, NITEM = C::NITEM, UTOK = C::UTOK;
  constexpr int NMA = C::NMA, NACA = C::NACA, NACR = C::NACR, NGW = C::NGW, SC = G::SC;
  constexpr int QHEAD = G::QHEAD, IMS = G::IMS, PLANE = G::PLANE, ITEM = G::ITEM;
  constexpr typename C::AccMap MA = C::make_map(false), MR = C::make_map(true);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full_bar[STAGES];
  __shared__ int pre_s[kMaxRows + 1];
  __shared__ int nt_s[kMaxRows + 1];        // work units per (row, head group), per row; then a sentinel
  __shared__ int sl_s[kMaxRows];
  __shared__ float red_s[2][QH][kThreads / 32];        // per-warp score maxima per head, by unit parity
  __shared__ float wsum_s[kThreads / 32][QH][NITEM + 1];
  __shared__ float off_s[QH][NITEM + 1];                // per head: offset sums per item; [NITEM] = softmax sum
  uint8_t* wimg = smem + STAGES * C::STAGE;
  uint32_t* qimg = reinterpret_cast<uint32_t*>(wimg + G::WIMG);
  const uint8_t* vzero = wimg + NITEM * ITEM;

  pdl_launch_dependents();   // the merge kernel may start staging R
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int H = a.g.Hq, HG = H / QH, B = a.batch;   // units run over (row, head group)
  const int Cn = gridDim.x, cta = blockIdx.x;

  for (int b = tid; b < B; b += kThreads) {
    const int n = clamp_len(a.seq_lens[b], a.g.Nmax);
    sl_s[b] = n;
    nt_s[b] = (n + UTOK - 1) / UTOK;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      pre_s[b] = acc;
      acc += HG * nt_s[b];
    }
    pre_s[B] = acc;
    nt_s[B] = 1;
  }
  __syncthreads();
  const int U = pre_s[B];
  if (U == 0) { pdl_wait(); return; }   // every row empty: the merge kernel writes the current V
  const Split split{U / Cn, U % Cn};
  const int u0 = split.start(cta), u1 = split.start(cta + 1);
  if (u0 >= u1) { pdl_wait(); return; }

  struct Cursor { int b, h, t; };   // row, head group, unit
  auto locate = [&](int u) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (pre_s[mid] <= u) lo = mid; else hi = mid - 1;
    }
    int rem = (int)(u - pre_s[lo]);
    return Cursor{lo, rem / nt_s[lo], rem % nt_s[lo]};
  };
  auto advance = [&](Cursor& c) {
    if (++c.t == nt_s[c.b]) {
      c.t = 0;
      if (++c.h == HG) {
        c.h = 0;
        do { ++c.b; } while (nt_s[c.b] == 0);
      }
    }
  };
  Cursor pc = locate(u0);
  const uint64_t pol = l2_evict_first_policy();
  auto unit_tiles = [&]() { return min(C::UT, (sl_s[pc.b] - pc.t * C::UT * kTile + kTile - 1) / kTile); };
  __shared__ int next_raw_s[C::UT];
  __shared__ int pu_s;
  auto fetch_pages = [&]() {
    const int nt = unit_tiles();
#pragma unroll
    for (int k = 0; k < C::UT; ++k) {
      if (k < nt)
        cp_async4(&next_raw_s[k], a.g.table + (size_t)pc.b * a.g.max_tiles + pc.t * C::UT + k);
      else
        next_raw_s[k] = 0;
    }
    cp_async_commit();
  };
  auto issue = [&](int stage) {
    if constexpr (PAGED) cp_async_wait_all();
    const int t0 = pc.t * C::UT;
    const int ntile = unit_tiles();
    const int kvh = (pc.h * QH) / a.g.qpk;   // the head group's KV head
    const uint8_t* region = PAGED ? a.base : a.base + a.g.region_offset(a.layer, a.group, pc.b, kvh);
    uint8_t* dst = smem + stage * C::STAGE;
    mbar_arrive_expect_tx(&full_bar[stage], (uint32_t)(ntile * C::SUB));
    for (int k = 0; k < ntile; ++k) {
      uint8_t* d = dst + k * C::SUB;
      const int tile = t0 + k;
      const uint8_t* blk = region;
      if constexpr (PAGED) {
        const int page = max(checked_page(a.g, next_raw_s[k], a.status), 0);
        blk = a.base + (((int64_t)a.layer * a.g.G + a.group) * a.g.num_pages + page) * a.g.page_bytes +
              (int64_t)kvh * a.g.head_block;
      }
      auto src = [&](bool anchor, int j, int kv) {
        if constexpr (PAGED)
          return blk + (anchor ? kv * C::A_TILE : 2 * C::A_TILE + (2 * j + kv) * C::R_TILE);
        else
          return region + (anchor ? a.g.anchor_plane(kv) : a.g.res_plane(j, kv)) +
                 (int64_t)tile * (anchor ? C::A_TILE : C::R_TILE);
      };
      bulk_g2s_hint(d, src(true, 0, 0), C::A_TILE, &full_bar[stage], pol);
      bulk_g2s_hint(d + C::A_TILE, src(true, 0, 1), C::A_TILE, &full_bar[stage], pol);
#pragma unroll
      for (int r = 0; r < NRES; ++r) {
        uint8_t* d0 = d + 2 * C::A_TILE + 2 * r * C::R_TILE;
        bulk_g2s_hint(d0, src(false, a.res0 + r, 0), C::R_TILE, &full_bar[stage], pol);
        bulk_g2s_hint(d0 + C::R_TILE, src(false, a.res0 + r, 1), C::R_TILE, &full_bar[stage], pol);
      }
    }
    advance(pc);
    if constexpr (PAGED)
      if (++pu_s < u1) fetch_pages();
  };

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&full_bar[s], 1);
    fence_mbar_init();
  }
  // the zero blocks: value B operands of unused columns, scoring B operands of idle lanes
  for (int i = tid; i < 64; i += kThreads) reinterpret_cast<uint32_t*>(wimg + NITEM * ITEM)[i] = 0u;
  for (int i = tid; i < QH * IMS; i += kThreads) qimg[(i / IMS) * QHEAD + kPackHeader + 8 * IMS + i % IMS] = 0u;
  __syncthreads();
  if (tid == 0) {
    if constexpr (PAGED) {
      pu_s = u0;
      fetch_pages();
    }
    for (int s = 0; s < STAGES && u0 + s < u1; ++s) issue(s);
  }
  Cursor cc = locate(u0);
  pdl_wait();   // the query packs of qprep_kernel are complete

  // ---- per-thread constants ----
  const int tk0 = 16 * warp + 4 * (gid >> 1) + (gid & 1), tau = warp >> 2, r0 = tk0 & (kTile - 1);
  int so4, so2;
  float sc4, sc2;
  int4_slot(tk0, so4, sc4);
  int2_slot(tk0, so2, sc2);
  // scoring B operands: lanes with (gid / 2) == tig read lane image (gid % 2) * 4 + tig, the others the zero image
  const int il = ((gid >> 1) == tig) ? (gid & 1) * 4 + tig : 8;
  const uint32_t* qlane = qimg + kPackHeader + il * IMS;
  const bool v_act = warp < C::VW;
  const int vc0 = 16 * warp + gid, vg = (16 * warp) / GS;
  const bool vb_lane = gid < G::NPL;   // lanes whose value B column belongs to a head

  // ---- per-segment state ----
  float m_run[QH], l_part[QH];
  float off_part[QH][1 + NRES][NGW];
  float acc_a[4] = {0.f, 0.f, 0.f, 0.f}, acc_r[4] = {0.f, 0.f, 0.f, 0.f};   // head tig's value accumulators (zero columns for tig >= QH)
  int cur_bh = -1;            // current (row, head group)
  bool aborted = false;
  int fail_u = 0;

  auto flush = [&](int bhg) {
    // offset sums and softmax denominators per head: over the lanes of a tig,
    // gathered to lane 0, which writes the warp's row with compile-time columns
#pragma unroll
    for (int h = 0; h < QH; ++h) {
#pragma unroll
      for (int j = 0; j <= NRES; ++j)
#pragma unroll
        for (int s = 0; s < NGW; ++s) {
          float x = off_part[h][j][s];
          for (int off = 4; off < 32; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float y = __shfl_sync(0xffffffffu, x, t);
            if (lane == 0 && 4 * s + t < NG) wsum_s[warp][h][j * NG + 4 * s + t] = y;
          }
        }
      float x = l_part[h];
      for (int off = 4; off < 32; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      if (lane == 0) wsum_s[warp][h][NITEM] = x;
    }
    __syncthreads();
    for (int i = tid; i < QH * (NITEM + 1); i += kThreads) {
      const int h = i / (NITEM + 1), k = i - h * (NITEM + 1);
      float x = 0.f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) x += wsum_s[w][h][k];
      off_s[h][k] = x;
    }
    __syncthreads();
    // partial rows (cta + bhg) * QH + h: distinct for every (CTA, head) of the call, as
    // cta + bhg is for every (CTA, head group) (a CTA's groups follow its predecessor's)
#pragma unroll
    for (int h = 0; h < QH; ++h)
      if (tid == h) {
        float* part = a.partials + ((size_t)(cta + bhg) * QH + h) * a.pstride;
        part[0] = m_run[h];
        part[1] = off_s[h][NITEM];
      }
    if (v_act && tig < QH) {   // lane tig holds head tig's accumulators
      float* part = a.partials + ((size_t)(cta + bhg) * QH + tig) * a.pstride;
      float oa = off_s[tig][vg], orr = 0.f;
#pragma unroll
      for (int r = 0; r < NRES; ++r) orr += off_s[tig][(1 + r) * NG + vg];
      part[2 + vc0] = fmaf(acc_a[0] + acc_a[1], 16777216.f, oa);
      part[2 + vc0 + 8] = fmaf(acc_a[2] + acc_a[3], 16777216.f, oa);
      if (NRES > 0) {
        part[2 + D + vc0] = fmaf(acc_r[0] + acc_r[1], 16777216.f, orr);
        part[2 + D + vc0 + 8] = fmaf(acc_r[2] + acc_r[3], 16777216.f, orr);
      }
    }
  };

  auto begin_segment = [&](int bhg) {
    // the group's query packs into shared memory (every warp is past the previous
    // unit's scoring products, the only readers of the images)
    const int b = bhg / HG, bh0 = b * H + (bhg - b * HG) * QH;
    constexpr int PW = kPackHeader + 8 * C::NIMG;   // words of a pack in use
    for (int i = tid; i < QH * PW; i += kThreads) {
      const int h = i / PW, w = i - h * PW;
      const uint32_t v = __ldcg(a.packs + (size_t)(bh0 + h) * kPackWords + w);
      const int e = w - kPackHeader;
      qimg[h * QHEAD + (w < kPackHeader ? w : kPackHeader + (e / C::NIMG) * IMS + e % C::NIMG)] = v;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < QH; ++h) {
      m_run[h] = -INFINITY;
      l_part[h] = 0.f;
#pragma unroll
      for (int j = 0; j <= NRES; ++j)
#pragma unroll
        for (int s = 0; s < NGW; ++s) off_part[h][j][s] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) { acc_a[i] = 0.f; acc_r[i] = 0.f; }
    cur_bh = bhg;
  };
  auto hdr = [&](int h, int k) { return __uint_as_float(qimg[h * QHEAD + k]); };

  for (int u = u0; u < u1; ++u, advance(cc)) {
    const int it = (int)(u - u0), stage = it % STAGES, buf = it & 1;
    const int bhg = cc.b * HG + cc.h;
    if (bhg != cur_bh) {
      if (cur_bh >= 0) flush(cur_bh);
      begin_segment(bhg);
    }
    const int n_valid = min(UTOK, sl_s[cc.b] - cc.t * UTOK);

    if (!mbar_wait_bounded(&full_bar[stage], (uint32_t)((it / STAGES) & 1))) aborted = true;

    const uint8_t* st = smem + stage * C::STAGE;
    const uint8_t* sub = st + tau * C::SUB;

    // ---- scores of tokens tk0, tk0 + 2 for every head of the group ----
    float sc0[QH], sc1[QH];
    {
      uint32_t wa0[C::WA], wa1[C::WA];
      const uint8_t* ak = sub + r0 * (D / 2) + tig * (D / 8);
      if constexpr (C::WA == 4) {
        const uint4 x0 = *reinterpret_cast<const uint4*>(ak);
        const uint4 x1 = *reinterpret_cast<const uint4*>(ak + 2 * (D / 2));
        wa0[0] = x0.x; wa0[1] = x0.y; wa0[2] = x0.z; wa0[3] = x0.w;
        wa1[0] = x1.x; wa1[1] = x1.y; wa1[2] = x1.z; wa1[3] = x1.w;
      } else {
#pragma unroll
        for (int k = 0; k < C::WA; ++k) {
          wa0[k] = *reinterpret_cast<const uint32_t*>(ak + 4 * k);
          wa1[k] = *reinterpret_cast<const uint32_t*>(ak + 2 * (D / 2) + 4 * k);
        }
      }
      const uint8_t* am = sub + C::A_CODES + r0 * NG * 2;
      float sa0[QH], sa1[QH];
#pragma unroll
      for (int h0 = 0; h0 < QH; h0 += SC) {
        float da[SC][NACA][4];
#pragma unroll
        for (int hh = 0; hh < SC; ++hh)
#pragma unroll
          for (int ac = 0; ac < NACA; ++ac) da[hh][ac][0] = da[hh][ac][1] = da[hh][ac][2] = da[hh][ac][3] = 0.f;
#pragma unroll
        for (int k = 0; k < C::WA; ++k) {
          uint32_t x0[4], x1[4];
          int4_f16(wa0[k], x0);
          int4_f16(wa1[k], x1);
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int j = 2 * k + jj;
#pragma unroll
            for (int hh = 0; hh < SC; ++hh) {
              const uint2 bb = *reinterpret_cast<const uint2*>(qlane + (h0 + hh) * QHEAD + 2 * j);
              mma16816(da[hh][MA.acc[j]], x0[2 * jj], x1[2 * jj], x0[2 * jj + 1], x1[2 * jj + 1], bb.x, bb.y);
            }
          }
        }
#pragma unroll
        for (int hh = 0; hh < SC; ++hh) {
          const int h = h0 + hh;
          const float sig = hdr(h, 0);
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int ac = 0; ac < NACA; ++ac) {
            const int g = C::ga(tig, MA.rep[ac]);
            const float2 m0 = meta2(am + g * 2), m1 = meta2(am + 2 * NG * 2 + g * 2);
            const bool own = (MA.own >> (4 * ac + tig)) & 1u;
            const float qo = hdr(h, 4 + g);
            s0 = fmaf(m0.x, (da[hh][ac][0] + da[hh][ac][1]) * sig, own ? fmaf(m0.y, qo, s0) : s0);
            s1 = fmaf(m1.x, (da[hh][ac][2] + da[hh][ac][3]) * sig, own ? fmaf(m1.y, qo, s1) : s1);
          }
          sa0[h] = s0;
          sa1[h] = s1;
        }
      }
#pragma unroll
      for (int h = 0; h < QH; ++h) { sc0[h] = sa0[h]; sc1[h] = sa1[h]; }
      if constexpr (NRES > 0) {
        float cp0 = 1.f, cp1 = 1.f, sr0[QH], sr1[QH];
#pragma unroll
        for (int h = 0; h < QH; ++h) sr0[h] = sr1[h] = 0.f;
#pragma unroll
        for (int r = 0; r < NRES; ++r) {
          const uint8_t* rk = sub + 2 * C::A_TILE + 2 * r * C::R_TILE;
          uint32_t w0[2] = {0u, 0u}, w1[2] = {0u, 0u};
          if (tig < C::TR) {
            const uint8_t* rr = rk + r0 * (D / 4) + tig * 8;
            const uint2 y0 = *reinterpret_cast<const uint2*>(rr);
            const uint2 y1 = *reinterpret_cast<const uint2*>(rr + 2 * (D / 4));
            w0[0] = y0.x; w0[1] = y0.y; w1[0] = y1.x; w1[1] = y1.y;
          }
          const uint8_t* rm = rk + C::R_CODES + r0 * NG * 2;
          float s0r[QH], s1r[QH];
#pragma unroll
          for (int h0 = 0; h0 < QH; h0 += SC) {
            float dr[SC][NACR][4];
#pragma unroll
            for (int hh = 0; hh < SC; ++hh)
#pragma unroll
              for (int ac = 0; ac < NACR; ++ac) dr[hh][ac][0] = dr[hh][ac][1] = dr[hh][ac][2] = dr[hh][ac][3] = 0.f;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              uint32_t x0[8], x1[8];
              int2_f16(w0[k], x0);
              int2_f16(w1[k], x1);
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const int j = 4 * k + jj;
#pragma unroll
                for (int hh = 0; hh < SC; ++hh) {
                  const uint2 bb =
                      *reinterpret_cast<const uint2*>(qlane + (h0 + hh) * QHEAD + 2 * NMA + 2 * j);
                  mma16816(dr[hh][MR.acc[j]], x0[2 * jj], x1[2 * jj], x0[2 * jj + 1], x1[2 * jj + 1], bb.x, bb.y);
                }
              }
            }
#pragma unroll
            for (int hh = 0; hh < SC; ++hh) {
              const int h = h0 + hh;
              float s0 = 0.f, s1 = 0.f;
              if (tig < C::TR) {
                const float sig = hdr(h, 1);
#pragma unroll
                for (int ac = 0; ac < NACR; ++ac) {
                  const int g = C::gr(tig, MR.rep[ac]);
                  const float2 m0 = meta2(rm + g * 2), m1 = meta2(rm + 2 * NG * 2 + g * 2);
                  const bool own = (MR.own >> (4 * ac + tig)) & 1u;
                  const float qo = hdr(h, 4 + NG + g);
                  s0 = fmaf(m0.x, (dr[hh][ac][0] + dr[hh][ac][1]) * sig, own ? fmaf(m0.y, qo, s0) : s0);
                  s1 = fmaf(m1.x, (dr[hh][ac][2] + dr[hh][ac][3]) * sig, own ? fmaf(m1.y, qo, s1) : s1);
                }
              }
              s0r[h] = s0;
              s1r[h] = s1;
            }
          }
          const uint8_t* rc = rk + C::R_CODES + C::META + r0 * 2;
          const float c0 = bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(rc));
          const float c1 = bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(rc + 4));
#pragma unroll
          for (int h = 0; h < QH; ++h) {
            sr0[h] = fmaf(cp0, s0r[h], sr0[h]);
            sr1[h] = fmaf(cp1, s1r[h], sr1[h]);
          }
          cp0 *= c0;
          cp1 *= c1;
        }
#pragma unroll
        for (int h = 0; h < QH; ++h) {
          sc0[h] = fmaf(cp0, sa0[h], sr0[h]);
          sc1[h] = fmaf(cp1, sa1[h], sr1[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < QH; ++h) {
        sc0[h] += __shfl_xor_sync(0xffffffffu, sc0[h], 1);
        sc1[h] += __shfl_xor_sync(0xffffffffu, sc1[h], 1);
        sc0[h] += __shfl_xor_sync(0xffffffffu, sc0[h], 2);
        sc1[h] += __shfl_xor_sync(0xffffffffu, sc1[h], 2);
      }
    }
    const bool ok0 = !aborted && tk0 < n_valid, ok1 = !aborted && tk0 + 2 < n_valid;
#pragma unroll
    for (int h = 0; h < QH; ++h) {
      if (!ok0) sc0[h] = -INFINITY;
      if (!ok1) sc1[h] = -INFINITY;
      float wmax = fmaxf(sc0[h], sc1[h]);
      for (int off = 4; off < 32; off <<= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));
      if (lane == 0) red_s[buf][h][warp] = wmax;
    }
    if (__syncthreads_or(aborted)) {                   // B1: per-warp score maxima are in red_s
      fail_u = u;
      aborted = true;
      if (tid == 0) atomicExch(&a.status[0], 1);
      break;
    }
    if (tid == 0 && it >= 1 && u - 1 + STAGES < u1) issue((it - 1) % STAGES);

    float alpha[QH], p0[QH], p1[QH];
#pragma unroll
    for (int h = 0; h < QH; ++h) {
      float m_tile = red_s[buf][h][0];
#pragma unroll
      for (int w = 1; w < kThreads / 32; ++w) m_tile = fmaxf(m_tile, red_s[buf][h][w]);
      const float m_new = fmaxf(m_run[h], m_tile);
      alpha[h] = ex2_fast(m_run[h] - m_new);
      m_run[h] = m_new;
      p0[h] = ex2_fast(sc0[h] - m_new);
      p1[h] = ex2_fast(sc1[h] - m_new);
      if (tig == 0) l_part[h] = fmaf(l_part[h], alpha[h], p0[h] + p1[h]);
#pragma unroll
      for (int j = 0; j <= NRES; ++j)
#pragma unroll
        for (int s = 0; s < NGW; ++s) off_part[h][j][s] *= alpha[h];
    }

    // ---- value weights of every head: p * coefficients * scale as f16 pieces ----
#pragma unroll
    for (int s = 0; s < NGW; ++s) {
      const int g = tig + 4 * s;
      if (g < NG) {
        float cc0 = 1.f, cc1 = 1.f;   // coefficients of the planes before the current one
#pragma unroll
        for (int r = 0; r < NRES; ++r) {
          const uint8_t* rv = sub + 2 * C::A_TILE + (2 * r + 1) * C::R_TILE + C::R_CODES;
          const float2 v0 = meta2(rv + r0 * NG * 2 + g * 2), v1 = meta2(rv + (r0 + 2) * NG * 2 + g * 2);
          uint8_t* im = wimg + ((1 + r) * NG + g) * ITEM + so2;
#pragma unroll
          for (int h = 0; h < QH; ++h) {
            const float w0 = p0[h] * cc0, w1 = p1[h] * cc1;
            if (ok0) off_part[h][1 + r][s] = fmaf(w0, v0.y, off_part[h][1 + r][s]);
            if (ok1) off_part[h][1 + r][s] = fmaf(w1, v1.y, off_part[h][1 + r][s]);
            uint32_t hi, lo;
            f16x2_pieces(ok0 ? w0 * v0.x * sc2 : 0.f, ok1 ? w1 * v1.x * sc2 : 0.f, hi, lo);
            *reinterpret_cast<uint32_t*>(im + (2 * h) * PLANE) = hi;
            *reinterpret_cast<uint32_t*>(im + (2 * h + 1) * PLANE) = lo;
          }
          const uint8_t* rc = rv + C::META + r0 * 2;
          if (ok0) cc0 *= bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(rc));
          if (ok1) cc1 *= bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(rc + 4));
        }
        const uint8_t* avm = sub + C::A_TILE + C::A_CODES;
        const float2 a0 = meta2(avm + r0 * NG * 2 + g * 2), a1 = meta2(avm + (r0 + 2) * NG * 2 + g * 2);
        uint8_t* im = wimg + g * ITEM + so4;
#pragma unroll
        for (int h = 0; h < QH; ++h) {
          const float w0 = p0[h] * cc0, w1 = p1[h] * cc1;
          if (ok0) off_part[h][0][s] = fmaf(w0, a0.y, off_part[h][0][s]);
          if (ok1) off_part[h][0][s] = fmaf(w1, a1.y, off_part[h][0][s]);
          uint32_t hi, lo;
          f16x2_pieces(ok0 ? w0 * a0.x * sc4 : 0.f, ok1 ? w1 * a1.x * sc4 : 0.f, hi, lo);
          *reinterpret_cast<uint32_t*>(im + (2 * h) * PLANE) = hi;
          *reinterpret_cast<uint32_t*>(im + (2 * h + 1) * PLANE) = lo;
        }
      }
    }
    __syncthreads();                                   // B2: the weight images are complete

    // ---- value products: channels vc0, vc0 + 8; column 2h + piece of head h ----
    if (v_act) {
      float al = alpha[0];   // the rescale of this lane's head (tig)
#pragma unroll
      for (int h = 1; h < QH; ++h)
        if (tig == h) al = alpha[h];
      const uint8_t* vb = vb_lane ? wimg + vg * ITEM + gid * PLANE + tig * 8 : vzero + tig * 8;
      float dv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int t2 = 0; t2 < C::UT; ++t2) {
        const uint8_t* av = st + t2 * C::SUB + C::A_TILE + vc0 * (kTile / 2) + tig * 8;
        const uint2 y0 = *reinterpret_cast<const uint2*>(av);
        const uint2 y1 = *reinterpret_cast<const uint2*>(av + 8 * (kTile / 2));
        const uint32_t w0[2] = {y0.x, y0.y}, w1[2] = {y1.x, y1.y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          uint32_t x0[4], x1[4];
          int4_f16(w0[e], x0);
          int4_f16(w1[e], x1);
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int m = 2 * (2 * t2 + e) + jj;
            const uint2 bb = *reinterpret_cast<const uint2*>(vb + m * 32);
            mma16816(dv, x0[2 * jj], x1[2 * jj], x0[2 * jj + 1], x1[2 * jj + 1], bb.x, bb.y);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) acc_a[i] = fmaf(acc_a[i], al, dv[i]);
      if constexpr (NRES > 0) {
        float dr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < NRES; ++r) {
          const uint8_t* vbr =
              vb_lane ? wimg + ((1 + r) * NG + vg) * ITEM + gid * PLANE + tig * 8 : vzero + tig * 8;
#pragma unroll
          for (int t2 = 0; t2 < C::UT; ++t2) {
            const uint8_t* rvp = st + t2 * C::SUB + 2 * C::A_TILE + (2 * r + 1) * C::R_TILE + vc0 * (kTile / 4) + tig * 4;
            const uint32_t y0 = *reinterpret_cast<const uint32_t*>(rvp);
            const uint32_t y1 = *reinterpret_cast<const uint32_t*>(rvp + 8 * (kTile / 4));
            uint32_t x0[8], x1[8];
            int2_f16(y0, x0);
            int2_f16(y1, x1);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int m = 4 * t2 + jj;
              const uint2 bb = *reinterpret_cast<const uint2*>(vbr + m * 32);
              mma16816(dr, x0[2 * jj], x1[2 * jj], x0[2 * jj + 1], x1[2 * jj + 1], bb.x, bb.y);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) acc_r[i] = fmaf(acc_r[i], al, dr[i]);
      }
    }
  }

  if (aborted) {
    if (tid == 0) {
      for (int v = fail_u; v < u1 && v < fail_u + STAGES; ++v)
        (void)mbar_wait_bounded(&full_bar[(v - u0) % STAGES], (uint32_t)(((v - u0) / STAGES) & 1));
      if constexpr (PAGED) cp_async_wait_all();
    }
    __syncthreads();
    return;
  }
  __syncthreads();
  if (cur_bh >= 0) flush(cur_bh);
}

template <int D, int GS, int NRES, bool PAGED, int QH>
cudaError_t launch_g(const DecodeArgs& a, int num_sms, cudaStream_t stream) {
  using G = GCfg<D, GS, NRES, QH>;
  auto k = decode_gqa_kernel<D, GS, NRES, PAGED, QH>;
  auto km = merge_kernel<D, (NRES > 0 ? 1 : 0), false>;
  size_t km_smem = NRES > 0 ? (size_t)D * D * sizeof(float) : 0;
  if (a.g.mode & RQ_MODE_HADAMARD) km_smem = 0;
  int km_threads = kMergeThreads, km_extra = 0;
  if constexpr (NRES == 0)
    if (a.kv_all) {
      km = merge_kernel<D, 0, true>;
      km_smem = TokenAppendSmem::bytes(a.g.P);
      km_threads = kAppendThreads;
      km_extra = a.batch * a.g.H;
    }
  constexpr size_t merge_smem = NRES > 0 ? (size_t)D * D * sizeof(float) : 0;
  // attributes per device, on the first call with the device current (as launch_t)
  static std::atomic<int> per_sm_dev[kMaxDevices];
  int dev = 0;
  cudaError_t e0 = cudaGetDevice(&dev);
  if (e0 != cudaSuccess) return e0;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int per_sm = per_sm_dev[dev].load(std::memory_order_acquire);
  if (per_sm == 0) {
    int optin = 0;
    e0 = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e0 != cudaSuccess) return e0;
    cudaFuncAttributes fa;
    e0 = cudaFuncGetAttributes(&fa, k);
    if (e0 != cudaSuccess) return e0;
    if ((size_t)G::SMEM + fa.sharedSizeBytes > (size_t)optin) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(merge_kernel<D, (NRES > 0 ? 1 : 0), false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)merge_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(qprep_kernel<D, GS, NRES>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(merge_kernel<D, (NRES > 0 ? 1 : 0), false>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             100);
    if (e != cudaSuccess) return e;
    if constexpr (NRES == 0) {
      e = cudaFuncSetAttribute(merge_kernel<D, 0, true>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return e;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, G::SMEM);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorNotSupported;
    per_sm = occ < G::MINB ? occ : G::MINB;
    per_sm_dev[dev].store(per_sm, std::memory_order_release);
  }
  const int grid = num_sms * per_sm;
  if (grid > kMaxContrib) return cudaErrorNotSupported;
  const int bhs = a.batch * a.g.Hq;
  cudaError_t e = launch_dependent(qprep_kernel<D, GS, NRES>, dim3(bhs), dim3(kPrepThreads), 0, stream, a);
  if (e != cudaSuccess) return e;
  e = launch_dependent(k, dim3(grid), dim3(kThreads), (size_t)G::SMEM, stream, a);
  if (e != cudaSuccess) return e;
  return launch_dependent(km, dim3(bhs + km_extra), dim3(km_threads), km_smem, stream, a, grid);
}

template <int D, int GS, bool PAGED, int QH>
cudaError_t launch_gq(const DecodeArgs& a, int num_sms, int nres, cudaStream_t stream) {
  if (nres == 0) return launch_g<D, GS, 0, PAGED, QH>(a, num_sms, stream);
  if (nres == 1) return launch_g<D, GS, 1, PAGED, QH>(a, num_sms, stream);
  return cudaErrorNotSupported;
}

template <int D, int GS>
cudaError_t launch_gd(const DecodeArgs& a, int num_sms, int nres, cudaStream_t stream) {
  if (a.qh == 4)
    return a.g.paged ? launch_gq<D, GS, true, 4>(a, num_sms, nres, stream)
                     : launch_gq<D, GS, false, 4>(a, num_sms, nres, stream);
  if (a.qh == 2)
    return a.g.paged ? launch_gq<D, GS, true, 2>(a, num_sms, nres, stream)
                     : launch_gq<D, GS, false, 2>(a, num_sms, nres, stream);
  return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_decode_gqa(const DecodeArgs& a, int num_sms, int nres, cudaStream_t stream) {
  const int d = a.g.d, gs = a.g.g;
  if (d == 128 && gs == 32) return launch_gd<128, 32>(a, num_sms, nres, stream);
  if (d == 128 && gs == 16) return launch_gd<128, 16>(a, num_sms, nres, stream);
  if (d == 96 && gs == 32) return launch_gd<96, 32>(a, num_sms, nres, stream);
  if (d == 96 && gs == 16) return launch_gd<96, 16>(a, num_sms, nres, stream);
  return cudaErrorNotSupported;
}

}  // namespace rq
