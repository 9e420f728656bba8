/*
 * Oracle for paged-latent MLA decode — TEST INFRASTRUCTURE ONLY.
 *
 * This file is the slow, obviously-correct CPU definition that the CUDA path is
 * checked against. Only the tests, the smoke check and the bench's CPU-baseline
 * leg may load it. It shares no code, header, table or constant generator with
 * the CUDA library: every codec, layout rule and formula below is written out
 * again from the sources it cites. All arithmetic is IEEE binary64 (C double),
 * except where a rounding decision must be taken in the kernel's precision
 * (the fp8 group scale choice, see mo_kv_write).
 *
 * Sources (page title, section):
 *  [vLLM-MLA]  "mla_attention.py · tduncan/Nvidia-Optimization-Stack-VLLM",
 *              module docstring, "Data-Movement Friendly Approach" (the absorbed
 *              MQA form: q = [ql_nope | q_pe] attends over [kv_c | k_pe] with
 *              V = kv_c) and "Compute Friendly Approach" (the MHA form).
 *  [vLLM-ctx]  same page, MLACommonMetadata (context_len / query_len / seq_len
 *              diagram) and neutralize_empty_context_partials (an empty partial
 *              is a zero output with an -inf lse).
 *  [vLLM-merge] same page, "Chunked Prefill" (merge_attn_states of two partial
 *              (output, lse) pairs).
 *  [HALOps-MLA] "MLA" API page of HALOps, mla_attention: kv_cache parameter
 *              (page = page_size rows of 448 e4m3 NoPE + 64 bf16 RoPE, then
 *              page_size 8-byte ue8m0 scale slots; page_bytes a multiple of the
 *              row size), attn_sink parameter (per-head logit added to the
 *              softmax denominator), and the supported-config paragraph (one
 *              ue8m0 scale per 64 NoPE elements, value dim 512).
 *              The same entry's kv_norm_weight, kv_eps, positions and freqs_real
 *              parameters and its step that normalises and rotates the kv row
 *              before the cache write define mo_kv_norm_rope.
 *  [sglang-FlashMLA] "Implementation:Sgl project Sglang Flash MLA", I/O Contract
 *              (q, k_cache, block_table, cache_seqlens, softmax_scale, causal,
 *              indices -> out, softmax_lse).
 *  OCP 8-bit floating point specification (E4M3: bias 7, no infinities,
 *  S.1111.111 is NaN, largest finite 448) and the OCP MX specification
 *  (E8M0 scale: 2^(b-127), 0xFF is NaN).
 *
 * Readings where the pages are silent:
 *  - lse is natural-log and covers keys only; the sink enters only the output
 *    denominator.
 *  - An empty candidate set gives out = 0 and lse = -inf, with or without sink.
 *  - Causal verify is bottom-right aligned: query token i of s_q sees context
 *    rows j <= L - s_q + i.
 *  - Sparse indices are request-local token positions; entries outside [0, L)
 *    are skipped; duplicates count as often as they appear.
 *  - The fp8 group exponent is the smallest e with 448 * 2^e >= max(amax, 1e-10),
 *    the eps being the fp32 value of 1e-10 (the kernel's precision).
 *  - RMSNorm covers the 512 latent elements with the mean of squares over 512;
 *    RoPE pairs are adjacent elements (interleaved), rotated by the table's
 *    (cos, sin); k_pe of the 576-wide rows is rotated but not normalised; the
 *    normalised row is rounded to bf16 once and then written as mo_kv_write
 *    writes a bf16 row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* Codecs                                                                     */
/* ------------------------------------------------------------------------- */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double mo_bf16_decode(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP E4M3 ("fn"): sign, 4-bit exponent (bias 7), 3-bit mantissa. E = 0 is
 * subnormal (M/8 * 2^-6); S.1111.111 is NaN; there is no infinity. */
double mo_e4m3_decode(uint8_t b) {
  int s = b >> 7, E = (b >> 3) & 0xF, M = b & 7;
  double v;
  if (E == 0xF && M == 7) return NAN;
  if (E == 0)
    v = ldexp((double)M, -9);                /* (M/8) * 2^(1-7) */
  else
    v = ldexp((double)(8 + M), E - 10);      /* (1 + M/8) * 2^(E-7) */
  return s ? -v : v;
}

/* Round-to-nearest-even onto the finite E4M3 grid, saturating to +-448
 * (the "satfinite" behaviour). Written as a search over the 127 non-negative
 * finite codes, which are increasing in value, so that it can be checked by
 * eye. Ties go to the code with an even mantissa (even code). */
uint8_t mo_e4m3_encode(double x) {
  uint8_t sign;
  double a, vlo, vhi;
  int lo, c;
  if (isnan(x)) return 0x7F;
  sign = signbit(x) ? 0x80 : 0x00;
  a = fabs(x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  lo = 0;
  for (c = 1; c <= 0x7E; ++c) {
    if (mo_e4m3_decode((uint8_t)c) <= a) lo = c;
    else break;
  }
  vlo = mo_e4m3_decode((uint8_t)lo);
  if (vlo == a) return (uint8_t)(sign | lo);
  vhi = mo_e4m3_decode((uint8_t)(lo + 1));
  if (a - vlo < vhi - a) return (uint8_t)(sign | lo);
  if (vhi - a < a - vlo) return (uint8_t)(sign | (lo + 1));
  return (uint8_t)(sign | ((lo & 1) ? lo + 1 : lo));
}

/* OCP MX E8M0 scale: 2^(b-127); 0xFF is NaN. */
double mo_ue8m0_decode(uint8_t b) {
  if (b == 0xFF) return NAN;
  return ldexp(1.0, (int)b - 127);
}

/* ------------------------------------------------------------------------- */
/* Paged row layouts                                                          */
/* ------------------------------------------------------------------------- */
/* layout 0: bf16 row [kv_c 512 | k_pe 64] = 1152 B; page = page_size rows.
 * layout 1: fp8 row [448 e4m3 NoPE | 64 bf16 RoPE] = 576 B; after the rows,
 *           page_size 8-byte scale slots (7 ue8m0 bytes + 1 zero pad byte);
 *           page_bytes = page_size * 584 rounded up to a multiple of 576.
 * layout 2: the same with 512 e4m3 NoPE (640 B rows, 8 scale bytes);
 *           page_bytes = page_size * 648 rounded up to a multiple of 640.
 * K has 576 (layouts 0, 2) or 512 (layout 1) elements; V is K[0:512]. */
int mo_layout_info(int layout, int page_size, int64_t* row_bytes, int64_t* page_bytes, int* dqk, int* nope,
                   int* n_scales) {
  int64_t rb, pb;
  if (page_size <= 0) return -1;
  switch (layout) {
    case 0: rb = 1152; pb = (int64_t)page_size * 1152; *dqk = 576; *nope = 512; *n_scales = 0; break;
    case 1: rb = 576; pb = (((int64_t)page_size * 584 + 575) / 576) * 576; *dqk = 512; *nope = 448; *n_scales = 7; break;
    case 2: rb = 640; pb = (((int64_t)page_size * 648 + 639) / 640) * 640; *dqk = 576; *nope = 512; *n_scales = 8; break;
    default: return -1;
  }
  *row_bytes = rb;
  *page_bytes = pb;
  return 0;
}

/* Decode one stored row into k[0:dqk] (fp64). Returns dqk, or -1. */
int mo_decode_row(const uint8_t* kv, int layout, int page_size, int64_t page, int offset, double* k) {
  int64_t rb, pb;
  int dqk, nope, ns, d;
  const uint8_t *row, *sc;
  uint16_t h;
  if (mo_layout_info(layout, page_size, &rb, &pb, &dqk, &nope, &ns) != 0) return -1;
  row = kv + page * pb + (int64_t)offset * rb;
  if (layout == 0) {
    for (d = 0; d < 576; ++d) {
      memcpy(&h, row + 2 * d, 2);
      k[d] = mo_bf16_decode(h);
    }
    return dqk;
  }
  sc = kv + page * pb + (int64_t)page_size * rb + (int64_t)offset * 8;
  for (d = 0; d < nope; ++d) k[d] = mo_e4m3_decode(row[d]) * mo_ue8m0_decode(sc[d / 64]);
  for (d = 0; d < 64; ++d) {
    memcpy(&h, row + nope + 2 * d, 2);
    k[nope + d] = mo_bf16_decode(h);
  }
  return dqk;
}

/* ------------------------------------------------------------------------- */
/* Attention over an explicit list of decoded rows                            */
/* ------------------------------------------------------------------------- */
/* [vLLM-MLA] MQA form: s_j = scale * <q, K_j>; softmax over j; out = sum_j p_j V_j
 * with V_j = K_j[0:dv]. lse = m + ln(sum_j e^(s_j - m)) over keys only; a sink
 * logit adds e^(sink - m) to the output denominator only [HALOps-MLA attn_sink].
 * Empty set: out = 0, lse = -inf [vLLM-ctx]. */
void mo_attend(const double* q, int dqk, const double* rows, int n_rows, int dv, double scale, int has_sink,
               double sink, double* out, double* lse) {
  double m, z, denom, *s;
  int j, d, v;
  for (v = 0; v < dv; ++v) out[v] = 0.0;
  if (n_rows <= 0) {
    *lse = -INFINITY;
    return;
  }
  s = (double*)malloc(sizeof(double) * (size_t)n_rows);
  m = -INFINITY;
  for (j = 0; j < n_rows; ++j) {
    double acc = 0.0;
    const double* kj = rows + (size_t)j * dqk;
    for (d = 0; d < dqk; ++d) acc += q[d] * kj[d];
    s[j] = scale * acc;
    if (s[j] > m) m = s[j];
  }
  z = 0.0;
  for (j = 0; j < n_rows; ++j) z += exp(s[j] - m);
  *lse = m + log(z);
  denom = z + (has_sink ? exp(sink - m) : 0.0);
  for (j = 0; j < n_rows; ++j) {
    double w = exp(s[j] - m) / denom;
    const double* kj = rows + (size_t)j * dqk;
    for (v = 0; v < dv; ++v) out[v] += w * kj[v];
  }
  free(s);
}

/* ------------------------------------------------------------------------- */
/* Paged decode                                                               */
/* ------------------------------------------------------------------------- */
/* [sglang-FlashMLA] I/O Contract: q [T = B*s_q, N, dqk] (bf16 bits), paged
 * k_cache addressed through block_table [B, max_pages], cache_seqlens [B],
 * optional indices [T, topk], causal flag; out [T, N, 512], lse [T, N].
 * If sel_t is non-NULL only the n_sel pairs (sel_t[i], sel_n[i]) are computed
 * and written to out[i*512], lse[i]; otherwise all T*N rows are.
 * Returns 0, or -1 on an out-of-range page reference. */
int mo_mla_decode(const uint16_t* q, const uint8_t* kv, int layout, int64_t num_pages, int page_size,
                  const int32_t* block_table, int max_pages, const int32_t* seqlens, int batch, int sq, int nheads,
                  double scale, const float* sink, const int32_t* indices, int topk, int causal,
                  const int32_t* sel_t, const int32_t* sel_n, int n_sel, double* out, double* lse, int nthreads) {
  int64_t rb, pb;
  int dqk, nope, ns;
  int T = batch * sq;
  int t, status = 0;
  int* want;       /* per token: number of selected heads (or nheads if all) */
  if (mo_layout_info(layout, page_size, &rb, &pb, &dqk, &nope, &ns) != 0) return -1;
  want = (int*)calloc((size_t)(T > 0 ? T : 1), sizeof(int));
  if (sel_t) {
    int i;
    for (i = 0; i < n_sel; ++i)
      if (sel_t[i] >= 0 && sel_t[i] < T) want[sel_t[i]]++;
  } else {
    for (t = 0; t < T; ++t) want[t] = nheads;
  }
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (t = 0; t < T; ++t) {
    int b = t / sq, i = t % sq, L = seqlens[b];
    int n_rows = 0, j, n, d, bad = 0, cap;
    int32_t* pos;
    double *rows, *qd;
    if (want[t] == 0) continue;
    /* candidate positions */
    cap = indices ? topk : (L > 0 ? L : 0);
    pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)(cap > 0 ? cap : 1));
    if (indices) {
      for (j = 0; j < topk; ++j) {
        int32_t idx = indices[(size_t)t * topk + j];
        if (idx >= 0 && idx < L) pos[n_rows++] = idx;
      }
    } else {
      int lim = L;
      if (causal) lim = L - sq + i + 1;
      if (lim > L) lim = L;
      for (j = 0; j < lim; ++j) pos[n_rows++] = j;
    }
    rows = (double*)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1) * dqk);
    for (j = 0; j < n_rows; ++j) {
      int blk = pos[j] / page_size, off = pos[j] % page_size;
      int64_t page;
      if (blk >= max_pages) { bad = 1; break; }
      page = block_table[(size_t)b * max_pages + blk];
      if (page < 0 || page >= num_pages) { bad = 1; break; }
      mo_decode_row(kv, layout, page_size, page, off, rows + (size_t)j * dqk);
    }
    qd = (double*)malloc(sizeof(double) * (size_t)dqk);
    if (!bad) {
      for (n = 0; n < nheads; ++n) {
        int slot = -1;
        if (sel_t) {
          int k2;
          for (k2 = 0; k2 < n_sel; ++k2)
            if (sel_t[k2] == t && sel_n[k2] == n) {
              slot = k2;
              for (d = 0; d < dqk; ++d) qd[d] = mo_bf16_decode(q[((size_t)t * nheads + n) * dqk + d]);
              mo_attend(qd, dqk, rows, n_rows, 512, scale, sink != NULL, sink ? (double)sink[n] : 0.0,
                        out + (size_t)slot * 512, lse + slot);
            }
        } else {
          slot = t * nheads + n;
          for (d = 0; d < dqk; ++d) qd[d] = mo_bf16_decode(q[((size_t)t * nheads + n) * dqk + d]);
          mo_attend(qd, dqk, rows, n_rows, 512, scale, sink != NULL, sink ? (double)sink[n] : 0.0,
                    out + (size_t)slot * 512, lse + slot);
        }
      }
    } else {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      status = -1;
    }
    free(qd);
    free(rows);
    free(pos);
  }
  free(want);
  return status;
}

/* ------------------------------------------------------------------------- */
/* Split combine                                                              */
/* ------------------------------------------------------------------------- */
/* [vLLM-merge] merge of partials: lse = ln sum_s e^(lse_s); out = sum_s
 * e^(lse_s - lse) o_s; a partial with lse = -inf carries no weight [vLLM-ctx].
 * The sink is applied once, after the merge: out *= 1 / (1 + e^(sink - lse))
 * [HALOps-MLA attn_sink]. All partials empty: out = 0, lse = -inf. */
void mo_combine(const double* part_out, const double* part_lse, int n_parts, int dv, int has_sink, double sink,
                double* out, double* lse) {
  double mx = -INFINITY, w, tot = 0.0, f;
  int s, v;
  for (v = 0; v < dv; ++v) out[v] = 0.0;
  for (s = 0; s < n_parts; ++s)
    if (part_lse[s] > mx) mx = part_lse[s];
  if (mx == -INFINITY) {
    *lse = -INFINITY;
    return;
  }
  for (s = 0; s < n_parts; ++s) tot += exp(part_lse[s] - mx);
  *lse = mx + log(tot);
  for (s = 0; s < n_parts; ++s) {
    w = exp(part_lse[s] - *lse);
    for (v = 0; v < dv; ++v) out[v] += w * part_out[(size_t)s * dv + v];
  }
  if (has_sink) {
    f = 1.0 / (1.0 + exp(sink - *lse));
    for (v = 0; v < dv; ++v) out[v] *= f;
  }
}

/* ------------------------------------------------------------------------- */
/* KV-row write                                                               */
/* ------------------------------------------------------------------------- */
/* Smallest e with 448 * 2^e >= a, found by exact power-of-two comparisons and
 * clamped to [-127, 127] so that e + 127 is a finite ue8m0 byte. */
int mo_group_exponent(double a) {
  int e;
  if (!(a <= 1e300)) return 127;   /* inf / nan */
  e = 0;
  while (e < 127 && ldexp(448.0, e) < a) ++e;
  while (e > -127 && ldexp(448.0, e - 1) >= a) --e;
  return e;
}

/* Write n rows (bf16 bits, [n, row_elems]) into the pages at slots[n]
 * (slot = page * page_size + offset; negative slots are skipped).
 * Layout 0: bit copy of 576 bf16. Layouts 1, 2: for each 64-element NoPE group,
 * amax = max(max |x|, eps) with eps = (float)1e-10, e = mo_group_exponent(amax),
 * scale byte = e + 127, code = E4M3 RNE-satfinite of x * 2^-e (exact product);
 * the 64 RoPE values are copied as bf16; the unused scale byte of layout 1 is 0.
 * A NaN element takes no part in amax and is stored as the NaN code 0x7F (what
 * mo_e4m3_encode gives for NaN); an infinite one makes amax infinite (e = 127).
 * Row elements: layout 0 -> 576, layout 1 -> 512 (448 | 64), layout 2 -> 576.
 * Returns 0, or -1 on an out-of-range slot. */
int mo_kv_write(const uint16_t* rows, const int32_t* slots, int n, uint8_t* kv, int layout, int64_t num_pages,
                int page_size) {
  int64_t rb, pb;
  int dqk, nope, ns, r;
  if (mo_layout_info(layout, page_size, &rb, &pb, &dqk, &nope, &ns) != 0) return -1;
  for (r = 0; r < n; ++r) {
    int64_t slot = slots[r], page;
    int off, g, d;
    const uint16_t* x = rows + (size_t)r * dqk;
    uint8_t *dst, *sc;
    if (slot < 0) continue;
    page = slot / page_size;
    off = (int)(slot % page_size);
    if (page >= num_pages) return -1;
    dst = kv + page * pb + (int64_t)off * rb;
    if (layout == 0) {
      memcpy(dst, x, 1152);
      continue;
    }
    sc = kv + page * pb + (int64_t)page_size * rb + (int64_t)off * 8;
    for (g = 0; g < 8; ++g) sc[g] = 0;
    for (g = 0; g < nope / 64; ++g) {
      double amax = 0.0, eps = (double)(float)1e-10;
      int e;
      for (d = 0; d < 64; ++d) {
        double v = fabs(mo_bf16_decode(x[g * 64 + d]));
        if (v > amax) amax = v;   /* the maximum over the numbers: a NaN element does not count */
      }
      if (amax < eps) amax = eps;
      e = mo_group_exponent(amax);
      sc[g] = (uint8_t)(e + 127);
      for (d = 0; d < 64; ++d) dst[g * 64 + d] = mo_e4m3_encode(ldexp(mo_bf16_decode(x[g * 64 + d]), -e));
    }
    memcpy(dst + nope, x + nope, 128);
  }
  return 0;
}

/* bfloat16 encoding of a binary64 value, rounded once to nearest (ties to even)
 * on the bfloat16 grid (8 significant bits, binary32 exponent range, subnormal
 * quantum 2^-133); overflow gives infinity. */
uint16_t mo_bf16_encode(double x) {
  if (isnan(x)) return 0x7FC0u;
  const uint16_t sign = signbit(x) ? 0x8000u : 0u;
  const double a = fabs(x);
  if (a == 0.0) return sign;
  int k;
  frexp(a, &k); /* a in [2^(k-1), 2^k) */
  int eb = k - 1;
  if (eb < -126) eb = -126;
  const double quantum = ldexp(1.0, eb - 7);
  const double y = nearbyint(a / quantum) * quantum;
  if (y >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
  const float fy = (float)y; /* exact: y lies on the bfloat16 grid */
  uint32_t u;
  memcpy(&u, &fy, sizeof u);
  return (uint16_t)((u >> 16) | sign);
}

/* RMSNorm + RoPE of new KV rows ([HALOps-MLA] mla_attention: the kv RMSNorm +
 * RoPE before the KV cache write; kv_norm_weight (gain of the 512 latent
 * elements), kv_eps, positions, and freqs_real: per position 32 interleaved
 * (cos, sin) pairs). Row i (bf16 bits, row_elems = 576 for layouts 0 and 2,
 * 512 for layout 1):
 *   y[d] = x[d] / sqrt(sum_{e<512} x[e]^2 / 512 + eps) * w[d]   for d < 512;
 *   RoPE pair i of the 64 RoPE elements, (c, s) = freqs[pos, 2i], freqs[pos, 2i+1]:
 *   (u, v) -> (u c - v s, u s + v c); layouts 0 and 2 rotate the raw elements
 *   512..575 (k_pe is not normalised), layout 1 rotates y[448..511];
 * the row is then rounded to bfloat16. Rows whose position lies outside
 * [0, max_pos) are left as zeros and return a count of them. */
int mo_kv_norm_rope(const uint16_t* raw, const int32_t* positions, const uint16_t* w, double eps, const float* freqs,
                    int max_pos, int n, int layout, uint16_t* out) {
  const int row_elems = layout == 1 ? 512 : 576;
  int bad = 0;
  for (int i = 0; i < n; ++i) {
    const uint16_t* x = raw + (size_t)i * row_elems;
    uint16_t* o = out + (size_t)i * row_elems;
    const int pos = positions[i];
    if (pos < 0 || pos >= max_pos) {
      memset(o, 0, sizeof(uint16_t) * row_elems);
      ++bad;
      continue;
    }
    double y[576];
    double ss = 0.0;
    for (int d = 0; d < 512; ++d) {
      const double v = mo_bf16_decode(x[d]);
      ss += v * v;
    }
    const double r = 1.0 / sqrt(ss / 512.0 + eps);
    for (int d = 0; d < 512; ++d) y[d] = mo_bf16_decode(x[d]) * r * mo_bf16_decode(w[d]);
    if (layout != 1)
      for (int d = 512; d < 576; ++d) y[d] = mo_bf16_decode(x[d]);
    const int rope0 = layout == 1 ? 448 : 512;
    const float* f = freqs + (size_t)pos * 64;
    for (int p = 0; p < 32; ++p) {
      const double c = f[2 * p], sn = f[2 * p + 1];
      const double u = y[rope0 + 2 * p], v = y[rope0 + 2 * p + 1];
      y[rope0 + 2 * p] = u * c - v * sn;
      y[rope0 + 2 * p + 1] = u * sn + v * c;
    }
    for (int d = 0; d < row_elems; ++d) o[d] = mo_bf16_encode(y[d]);
  }
  return bad;
}

/* Value up-projection ([vLLM-MLA] _v_up_proj: the (N, B, L) latent output times
 * W_UV (N, L, V)): o[t, n, v] = bf16(sum_l x[t, n, l] * w[n, l, v]) for x the
 * bf16 latent rows [T, N, 512] and w bf16 [N, 512, dv]. */
void mo_v_up(const uint16_t* x, const uint16_t* w, int T, int N, int dv, uint16_t* o) {
  for (int t = 0; t < T; ++t)
    for (int n = 0; n < N; ++n)
      for (int v = 0; v < dv; ++v) {
        double acc = 0.0;
        for (int l = 0; l < 512; ++l)
          acc += mo_bf16_decode(x[((size_t)t * N + n) * 512 + l]) * mo_bf16_decode(w[((size_t)n * 512 + l) * dv + v]);
        o[((size_t)t * N + n) * dv + v] = mo_bf16_encode(acc);
      }
}

/* Inverse RoPE of attention output rows ([HALOps-MLA] mla_output_proj, which undoes
 * the rotation of O): for each bf16 row [512], elements [rope0, rope0 + 64) hold 32 interleaved
 * pairs (u, v) rotated by the position's angle; they are rotated back,
 * (u, v) -> (u c + v s, v c - u s) with (c, s) = freqs[pos, 2i], freqs[pos, 2i+1],
 * and rounded to bf16. Rows with a position outside [0, max_pos) are copied. */
void mo_inv_rope(const uint16_t* x, const int32_t* positions, const float* freqs, int max_pos, int rope0, int nrows,
                 uint16_t* out) {
  for (int r = 0; r < nrows; ++r) {
    const uint16_t* xr = x + (size_t)r * 512;
    uint16_t* o = out + (size_t)r * 512;
    memcpy(o, xr, 512 * sizeof(uint16_t));
    const int pos = positions[r];
    if (pos < 0 || pos >= max_pos) continue;
    const float* f = freqs + (size_t)pos * 64;
    for (int i = 0; i < 32; ++i) {
      const double c = f[2 * i], sn = f[2 * i + 1];
      const double u = mo_bf16_decode(xr[rope0 + 2 * i]), v = mo_bf16_decode(xr[rope0 + 2 * i + 1]);
      o[rope0 + 2 * i] = mo_bf16_encode(u * c + v * sn);
      o[rope0 + 2 * i + 1] = mo_bf16_encode(v * c - u * sn);
    }
  }
}

/* Sliding-window runs ([HALOps-MLA] mla_attention_plan): token t's window is
 * kv_indices[t, 0 .. len), len = lengths[t] clamped to [0, topk] (topk when lengths is
 * NULL). Walking it in order, a run continues while the next slot is the previous one
 * plus step and on the same page (slot / page_size); a window of more than two runs is
 * cut to its first row. Output (slot0, len0, slot1, rows) per token, each run given by its
 * lowest slot (row g < len0 -> slot0 + g, else slot1 + g - len0); an empty window gives
 * zeros; a single run gives slot1 = slot0 + len0. */
void mo_swa_plan(const int32_t* idx, const int32_t* lengths, int T, int topk, int page_size, int step, int32_t* runs) {
  for (int t = 0; t < T; ++t) {
    const int32_t* w = idx + (size_t)t * topk;
    int32_t* o = runs + (size_t)t * 4;
    int len = lengths ? lengths[t] : topk;
    if (len < 0) len = 0;
    if (len > topk) len = topk;
    if (len == 0) {
      o[0] = o[1] = o[2] = o[3] = 0;
      continue;
    }
    /* split the window into maximal runs */
    int starts[3], counts[3], n = 0;
    for (int g = 0; g < len && n <= 2; ++g) {
      const int cont = g > 0 && w[g] == w[g - 1] + step &&
                       (int)floor((double)w[g] / page_size) == (int)floor((double)w[g - 1] / page_size);
      if (cont) {
        counts[n - 1] += 1;
      } else {
        if (n == 2) {
          n = 3;
          break;
        }
        starts[n] = w[g];
        counts[n] = 1;
        n += 1;
      }
    }
    if (n > 2) {
      o[0] = w[0];
      o[1] = 1;
      o[2] = w[0];
      o[3] = 1;
      continue;
    }
    const int lo0 = step > 0 ? starts[0] : starts[0] - (counts[0] - 1);
    o[0] = lo0;
    o[1] = counts[0];
    o[2] = n == 2 ? (step > 0 ? starts[1] : starts[1] - (counts[1] - 1)) : lo0 + counts[0];
    o[3] = len;
  }
}

/* Decoded rows 0..L-1 of one request (block_table row given) -> out [L, dqk]. */
int mo_kv_gather(const uint8_t* kv, int layout, int64_t num_pages, int page_size, const int32_t* bt_row,
                 int max_pages, int L, double* out) {
  int64_t rb, pb;
  int dqk, nope, ns, j;
  if (mo_layout_info(layout, page_size, &rb, &pb, &dqk, &nope, &ns) != 0) return -1;
  for (j = 0; j < L; ++j) {
    int blk = j / page_size;
    int64_t page;
    if (blk >= max_pages) return -1;
    page = bt_row[blk];
    if (page < 0 || page >= num_pages) return -1;
    mo_decode_row(kv, layout, page_size, page, j % page_size, out + (size_t)j * dqk);
  }
  return 0;
}

/* Sparse prefill ([sglang-FlashMLA] Signature and I/O Contract of flash_mla_sparse_fwd:
 * q, kv, indices, sm_scale, d_v = 512 -> out, max_logits, lse). kv is one unpaged run of
 * s_kv latent rows (bf16 bits [s_kv, 576]); token t's candidate rows are the entries of
 * indices[t, 0 .. topk) inside [0, s_kv) (others are skipped; duplicates count twice).
 * For each (t, n): the attention of q[t, n] over those rows with V = row[0 : 512]
 * (mo_attend: out, natural-log lse over the keys), and max_logits = the largest scaled
 * score sm_scale * <q, K_j> (-inf when there is no candidate; out = 0, lse = -inf then). */
void mo_sparse_prefill(const uint16_t* q, const uint16_t* kv, int s_kv, const int32_t* indices, int topk, int T,
                       int nheads, double scale, double* out, double* max_logits, double* lse, int nthreads) {
  int t;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (t = 0; t < T; ++t) {
    int n_rows = 0, j, d, n;
    double* rows = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1) * 576);
    double qd[576];
    for (j = 0; j < topk; ++j) {
      const int32_t idx = indices[(size_t)t * topk + j];
      if (idx < 0 || idx >= s_kv) continue;
      for (d = 0; d < 576; ++d) rows[(size_t)n_rows * 576 + d] = mo_bf16_decode(kv[(size_t)idx * 576 + d]);
      ++n_rows;
    }
    for (n = 0; n < nheads; ++n) {
      const size_t o = (size_t)t * nheads + n;
      double mx = -INFINITY;
      for (d = 0; d < 576; ++d) qd[d] = mo_bf16_decode(q[o * 576 + d]);
      for (j = 0; j < n_rows; ++j) {
        double acc = 0.0;
        for (d = 0; d < 576; ++d) acc += qd[d] * rows[(size_t)j * 576 + d];
        if (scale * acc > mx) mx = scale * acc;
      }
      max_logits[o] = mx;
      mo_attend(qd, 576, rows, n_rows, 512, scale, 0, 0.0, out + o * 512, lse + o);
    }
    free(rows);
  }
}
