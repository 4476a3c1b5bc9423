/*
 * CPU oracle for the NVFP4 weight-only (W4A16) MoE decode layer.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, plain reference that the
 * CUDA library is checked against. Only the test-suite, the smoke check and
 * the bench's CPU-baseline leg may load it. It shares no code, header, table
 * or constant generator with the CUDA library.
 *
 * Sources (page title, section):
 *  - "Lynn Engine: native LLM inference engine for NVIDIA Blackwell" (zingnex
 *    write-up), section "core features / 1. native NVFP4": weights are 4-bit
 *    E2M1, activations stay bf16 (W4A16); packed weights are consumed directly.
 *  - lynn-engine README (GitHub), stage notes P1 (packed E2M1 + per-16 FP16
 *    scale matvec), P28/P29 (gate/up + SiLU -> [top_k, I] intermediate; down +
 *    routing-weighted sum -> [H]), P45 (one-call active MoE contract), P52/P89
 *    (per-16 block scales consumed exactly, one scale per 16 K elements).
 *  - lynn-engine tutorials index, row 06 (MoE router): softmax over all experts,
 *    then top-k, then renormalise; the shared expert is gated by a sigmoid.
 *  - lynn-engine tutorials index, "Qwen 3.6 35B-A3B" config block: hidden 2048,
 *    256 experts, 8 per token, shared expert with sigmoid gate.
 *
 * Arithmetic: every reduction and every activation is in fp64. Element values
 * are converted exactly (bf16 and the decoded NVFP4 products are exact in fp64).
 * The packer is specified in fp32 IEEE round-to-nearest-even steps so that its
 * bytes are reproducible bit for bit; build without fast-math and with
 * -ffp-contract=off.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - E2M1 magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}, bit 3 = sign; rounding is
 *    round-to-nearest-even on that grid, saturating at 6; the sign of w is kept
 *    even when the magnitude rounds to 0.
 *  - element 2j in the low nibble, element 2j+1 in the high nibble of byte j;
 *    packed [N, K/2] and scales [N, K/16], both row-major.
 *  - E4M3 scales: tensor scale s_t = amax(W) / (6 * 448) (1 if amax = 0);
 *    block code e = E4M3_rne_satfinite((amax_b / 6) / s_t).
 *    FP16 scales: s_t = 1, block code e = FP16_rne_satfinite(amax_b / 6).
 *    Each element is quantised against the decoded scale e * s_t.
 *  - top-k order: larger probability first, lower expert index on exact ties.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_SCALE_E4M3 0
#define ORC_SCALE_FP16 1
#define ORC_SCALE_FP32 2    /* fp32 block scale per 16 elements, tensor scale 1 (README P52) */
#define ORC_SCALE_UE8M0 3   /* power-of-two E8M0 scale per 32 elements, tensor scale 1 (README P17/P18) */

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_NONFINITE 2
#define ORC_ERR_MISSING_EXPERT 3

/* ------------------------------------------------------------------ formats */

/* E2M1 magnitude of a 3-bit code: subnormal for exponent 0 (step 0.5), normal
 * (1 + m/2) * 2^(e-1) otherwise. */
double orc_e2m1_decode(int code) {
    int mag = code & 7;
    int e = mag >> 1, m = mag & 1;
    double v = (e == 0) ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
    return (code & 8) ? -v : v;
}

/* Round an fp32 value to the E2M1 grid: nearest, ties to the even mantissa,
 * saturate at 6. Returns the 4-bit code. */
int orc_e2m1_encode(float v) {
    int sign = signbit(v) ? 8 : 0;
    float a = fabsf(v);
    int mag;
    if (!(a < 6.0f)) {
        mag = 7; /* saturate (also +inf; NaN is rejected by the caller) */
    } else if (a < 1.0f) {
        float q = rintf(a * 2.0f);          /* exact scaling, rint = ties-to-even */
        mag = (int)q;                        /* 0, 1 or 2 (2 == 1.0 == code 2) */
    } else {
        int ex;
        frexpf(a, &ex);                      /* a = f * 2^ex, f in [0.5, 1) */
        int E = ex - 1;                      /* a in [2^E, 2^(E+1)), E in 0..2 */
        float q = rintf(ldexpf(a, 1 - E));   /* units of 2^(E-1): 2..4 */
        int qi = (int)q;
        if (qi == 4) { E += 1; qi = 2; }
        if (E > 2) { mag = 7; }              /* 8 is not representable: saturate to 6 */
        else mag = ((E + 1) << 1) | (qi - 2);
    }
    return sign | mag;
}

/* E4M3 (finite variant: no infinity, 0x7F is NaN, max 448). */
double orc_e4m3_decode(int byte) {
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return s ? -v : v;
}

/* Round an fp32 value to E4M3: nearest, ties to even, saturate to +-448. */
int orc_e4m3_encode(float v) {
    int s = signbit(v) ? 0x80 : 0;
    float a = fabsf(v);
    if (!(a <= 448.0f)) return s | 0x7E;     /* satfinite (NaN rejected upstream) */
    if (a < 0.015625f) {                     /* below 2^-6: subnormal step 2^-9 */
        int q = (int)rintf(ldexpf(a, 9));    /* 0..8; 8 is the first normal */
        if (q == 8) return s | (1 << 3);
        return s | q;
    }
    int ex;
    frexpf(a, &ex);
    int E = ex - 1;                          /* a in [2^E, 2^(E+1)), E >= -6 */
    int q = (int)rintf(ldexpf(a, 3 - E));    /* 8..16 in units of 2^(E-3) */
    if (q == 16) { E += 1; q = 8; }
    int eb = E + 7;
    int m = q - 8;
    if (eb > 15 || (eb == 15 && m == 7)) return s | 0x7E;
    return s | (eb << 3) | m;
}

double orc_fp16_decode(int bits) {
    int s = (bits >> 15) & 1, e = (bits >> 10) & 31, m = bits & 1023;
    double v;
    if (e == 31) return m ? NAN : (s ? -INFINITY : INFINITY);
    if (e == 0) v = ldexp((double)m, -24);
    else v = (1.0 + m / 1024.0) * ldexp(1.0, e - 15);
    return s ? -v : v;
}

/* Round an fp32 value to binary16: nearest, ties to even, saturate to +-65504. */
int orc_fp16_encode(float v) {
    int s = signbit(v) ? 0x8000 : 0;
    float a = fabsf(v);
    if (!(a <= 65504.0f)) return s | 0x7BFF;
    if (a < 6.103515625e-05f) {              /* below 2^-14: subnormal step 2^-24 */
        int q = (int)rintf(ldexpf(a, 24));   /* 0..1024; 1024 is the first normal */
        return s | q;                        /* q == 1024 encodes e=1, m=0 */
    }
    int ex;
    frexpf(a, &ex);
    int E = ex - 1;
    int q = (int)rintf(ldexpf(a, 10 - E));   /* 1024..2048 */
    if (q == 2048) { E += 1; q = 1024; }
    int eb = E + 15;
    if (eb > 30) return s | 0x7BFF;
    return s | (eb << 10) | (q - 1024);
}

static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* E8M0 (OCP MX shared scale): 2^(byte - 127); 0xFF is NaN. */
double orc_e8m0_decode(int byte) {
    if ((byte & 0xFF) == 0xFF) return NAN;
    return ldexp(1.0, (byte & 0xFF) - 127);
}

/* Elements per scale block of a scale kind. */
static int block_elems(int kind) { return kind == ORC_SCALE_UE8M0 ? 32 : 16; }

static double scale_value(const void* scales, int kind, size_t idx) {
    if (kind == ORC_SCALE_E4M3) return orc_e4m3_decode(((const uint8_t*)scales)[idx]);
    if (kind == ORC_SCALE_FP32) return (double)((const float*)scales)[idx];
    if (kind == ORC_SCALE_UE8M0) return orc_e8m0_decode(((const uint8_t*)scales)[idx]);
    return orc_fp16_decode(((const uint16_t*)scales)[idx]);
}

/* -------------------------------------------------------------------- pack */

/* Quantise fp32 W[N,K] (row-major) to NVFP4: packed [N,K/2], scales [N,K/B] (B = 16, or
 * 32 for UE8M0), one fp32 tensor scale. Per scale kind:
 *   E4M3   s_t = amax(W)/(6*448) (1 if amax = 0); block code = E4M3_rne_satfinite((amax_b/6)/s_t)
 *   FP16   s_t = 1; block code = FP16_rne_satfinite(amax_b/6)
 *   FP32   s_t = 1; block scale = amax_b/6 (one fp32 division)
 *   UE8M0  s_t = 1; block exponent = floor(log2(amax_b)) - 2 (the OCP MX rule: the largest
 *          power of two of E2M1 is 2^2), clamped to the E8M0 range [-127, 127]; 0 for amax_b = 0
 * and every element becomes the E2M1 code nearest to w / (decoded block scale * s_t). */
int orc_pack(const float* w, int N, int K, int kind, uint8_t* packed, void* scales,
             float* tensor_scale) {
    if (kind != ORC_SCALE_E4M3 && kind != ORC_SCALE_FP16 && kind != ORC_SCALE_FP32 && kind != ORC_SCALE_UE8M0)
        return ORC_ERR_ARG;
    const int B = block_elems(kind);
    if (N < 0 || K < 0 || K % B != 0) return ORC_ERR_ARG;
    size_t total = (size_t)N * K;
    float amax_t = 0.0f;
    for (size_t i = 0; i < total; ++i) {
        if (!isfinite(w[i])) return ORC_ERR_NONFINITE;
        float a = fabsf(w[i]);
        if (a > amax_t) amax_t = a;
    }
    float s_t = 1.0f;
    if (kind == ORC_SCALE_E4M3 && amax_t > 0.0f) s_t = amax_t / 2688.0f;
    *tensor_scale = s_t;
    int nb = K / B;
    for (int n = 0; n < N; ++n) {
        for (int b = 0; b < nb; ++b) {
            const float* blk = w + (size_t)n * K + (size_t)b * B;
            float amax_b = 0.0f;
            for (int i = 0; i < B; ++i) {
                float a = fabsf(blk[i]);
                if (a > amax_b) amax_b = a;
            }
            float r = amax_b / 6.0f;
            float dec;
            size_t sidx = (size_t)n * nb + b;
            if (kind == ORC_SCALE_E4M3) {
                int e = orc_e4m3_encode(r / s_t);
                ((uint8_t*)scales)[sidx] = (uint8_t)e;
                dec = (float)orc_e4m3_decode(e) * s_t;
            } else if (kind == ORC_SCALE_FP16) {
                int e = orc_fp16_encode(r);
                ((uint16_t*)scales)[sidx] = (uint16_t)e;
                dec = (float)orc_fp16_decode(e) * s_t;
            } else if (kind == ORC_SCALE_FP32) {
                ((float*)scales)[sidx] = r;
                dec = r;
            } else {
                int ex = 0;
                if (amax_b > 0.0f) {
                    int fe;
                    frexpf(amax_b, &fe);         /* amax_b = f * 2^fe, f in [0.5, 1) */
                    ex = (fe - 1) - 2;           /* floor(log2(amax_b)) - 2 */
                    if (ex < -127) ex = -127;
                    if (ex > 127) ex = 127;
                }
                ((uint8_t*)scales)[sidx] = (uint8_t)(ex + 127);
                dec = ldexpf(1.0f, ex);
            }
            uint8_t* out = packed + (size_t)n * (K / 2) + (size_t)b * (B / 2);
            for (int j = 0; j < B / 2; ++j) {
                int lo = 0, hi = 0;
                if (dec > 0.0f) {
                    lo = orc_e2m1_encode(blk[2 * j] / dec);
                    hi = orc_e2m1_encode(blk[2 * j + 1] / dec);
                }
                out[j] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    return ORC_OK;
}

/* ----------------------------------------------------------------- dequant */

/* W[n,k] = E2M1(code) * scale(n, k/16) * tensor_scale, in fp64 (exact). */
void orc_dequant(const uint8_t* packed, const void* scales, float tensor_scale, int kind,
                 int N, int K, double* out) {
    const int B = block_elems(kind);
    int nb = K / B;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            uint8_t byte = packed[(size_t)n * (K / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            out[(size_t)n * K + k] = orc_e2m1_decode(code) *
                                     scale_value(scales, kind, (size_t)n * nb + k / B) *
                                     (double)tensor_scale;
        }
}

/* Dot product of dequantised row n with an fp64 vector v[K]. */
static double row_dot(const uint8_t* packed, const void* scales, float ts, int kind, int n,
                      int K, const double* v) {
    const int B = block_elems(kind);
    int nb = K / B;
    double acc = 0.0;
    for (int k = 0; k < K; ++k) {
        uint8_t byte = packed[(size_t)n * (K / 2) + k / 2];
        int code = (k & 1) ? (byte >> 4) : (byte & 15);
        double wv = orc_e2m1_decode(code) * scale_value(scales, kind, (size_t)n * nb + k / B) *
                    (double)ts;
        acc += wv * v[k];
    }
    return acc;
}

/* ------------------------------------------------------------- dense GEMV */

/* y[t,n] = sum_k W[n,k] * x[t,k]; x is bf16 [T,K], y fp64 [T,N]. */
void orc_gemv(const uint8_t* packed, const void* scales, float ts, int kind, int N, int K,
              const uint16_t* x, int T, double* y) {
    double* xv = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) xv[k] = bf16_to_double(x[(size_t)t * K + k]);
        for (int n = 0; n < N; ++n) y[(size_t)t * N + n] = row_dot(packed, scales, ts, kind, n, K, xv);
    }
    free(xv);
}

/* ------------------------------------------------------------------ router */

/* logits[t,e] = sum_h x[t,h] * Wg[e,h], both bf16. */
void orc_router_logits(const uint16_t* x, int T, int H, const uint16_t* wg, int E,
                       double* logits) {
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += bf16_to_double(x[(size_t)t * H + h]) * bf16_to_double(wg[(size_t)e * H + h]);
            logits[(size_t)t * E + e] = acc;
        }
}

/* p = softmax over all E logits; keep the k largest p, in that order; w =
 * p_topk / sum(p_topk). probs (nullable) receives p. softmax is monotone in the
 * logits, so equal p with different logits (exp underflowing to 0, or rounding
 * to the same double) are ordered by the logits: the top-k of p as defined, not
 * an artefact of fp64 range. Equal logits: lower index first. */
int orc_route(const double* logits, int T, int E, int k, int32_t* ids, double* w,
              double* probs) {
    if (k < 1 || k > E) return ORC_ERR_ARG;
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    char* taken = (char*)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const double* l = logits + (size_t)t * E;
        double mx = l[0];
        for (int e = 1; e < E; ++e) if (l[e] > mx) mx = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) { p[e] = exp(l[e] - mx); z += p[e]; }
        for (int e = 0; e < E; ++e) p[e] /= z;
        if (probs) memcpy(probs + (size_t)t * E, p, sizeof(double) * (size_t)E);
        memset(taken, 0, (size_t)E);
        double sum = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || p[e] > p[best] || (p[e] == p[best] && l[e] > l[best]))
                    best = e;   /* strict: lower index wins exact ties */
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
            w[(size_t)t * k + j] = p[best];
            sum += p[best];
        }
        for (int j = 0; j < k; ++j) w[(size_t)t * k + j] /= sum;
    }
    free(p);
    free(taken);
    return ORC_OK;
}

/* ---------------------------------------------------------------- experts */

static double silu(double z) { return z / (1.0 + exp(-z)); }
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* One NVFP4 weight matrix as the oracle sees it. */
typedef struct {
    const uint8_t* packed;
    const void* scales;
    float tensor_scale;
} orc_mat;

/* out[H] = Down( silu(Gate x) * (Up x) ) for one token; x fp64 [H]. */
static void swiglu_expert(const orc_mat* g, const orc_mat* u, const orc_mat* d, int kind, int H,
                          int I, const double* x, double* h_tmp, double* out) {
    for (int i = 0; i < I; ++i) {
        double gv = row_dot(g->packed, g->scales, g->tensor_scale, kind, i, H, x);
        double uv = row_dot(u->packed, u->scales, u->tensor_scale, kind, i, H, x);
        h_tmp[i] = silu(gv) * uv;
    }
    for (int n = 0; n < H; ++n) out[n] = row_dot(d->packed, d->scales, d->tensor_scale, kind, n, I, h_tmp);
}

/* Public single-expert SwiGLU (used by the reduction pins). */
void orc_swiglu(const uint8_t* gp, const void* gs, float gts, const uint8_t* up, const void* us,
                float uts, const uint8_t* dp, const void* ds, float dts, int kind, int H, int I,
                const uint16_t* x, int T, double* y) {
    orc_mat g = {gp, gs, gts}, u = {up, us, uts}, d = {dp, ds, dts};
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    double* ht = (double*)malloc(sizeof(double) * (size_t)(I > 0 ? I : 1));
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h) xv[h] = bf16_to_double(x[(size_t)t * H + h]);
        swiglu_expert(&g, &u, &d, kind, H, I, xv, ht, y + (size_t)t * H);
    }
    free(xv);
    free(ht);
}

/*
 * The MoE layer for T tokens:
 *   logits = x Wg^T;  p = softmax(logits);  (ids, w) = renormalised top-k of p
 *   y[t] = sum_j w[t,j] * SwiGLU_{ids[t,j]}(x[t]) + sigmoid(gs . x[t]) * SwiGLU_shared(x[t])
 * Expert matrices are passed per expert as arrays of E pointers; an expert that
 * routing selects but whose pointer is NULL makes the call fail with
 * ORC_ERR_MISSING_EXPERT (callers only materialise the experts they need).
 * If force_ids is non-NULL it replaces the top-k selection (weights are then
 * p[id] renormalised over the forced set) - used for near-tie tokens.
 * y: fp64 [T,H]; ids_out [T,k], w_out [T,k], sig_out [T] (all nullable).
 */
int orc_moe_layer(int H, int E, int k, int I, int Is, int kind, const uint16_t* x, int T,
                  const uint16_t* router_w, const uint16_t* sh_gate_vec,
                  const uint8_t* const* g_packed, const void* const* g_scales, const float* g_ts,
                  const uint8_t* const* u_packed, const void* const* u_scales, const float* u_ts,
                  const uint8_t* const* d_packed, const void* const* d_scales, const float* d_ts,
                  const uint8_t* sg_packed, const void* sg_scales, float sg_ts,
                  const uint8_t* su_packed, const void* su_scales, float su_ts,
                  const uint8_t* sd_packed, const void* sd_scales, float sd_ts,
                  const int32_t* force_ids, double* y, int32_t* ids_out, double* w_out,
                  double* sig_out) {
    if (H <= 0 || E <= 0 || k < 1 || k > E || I <= 0 || Is < 0 || T < 0) return ORC_ERR_ARG;
    int rc = ORC_OK;
    double* logits = (double*)malloc(sizeof(double) * (size_t)E * (T > 0 ? T : 1));
    double* probs = (double*)malloc(sizeof(double) * (size_t)E * (T > 0 ? T : 1));
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)k * (T > 0 ? T : 1));
    double* w = (double*)malloc(sizeof(double) * (size_t)k * (T > 0 ? T : 1));
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    int imax = I > Is ? I : Is;
    double* ht = (double*)malloc(sizeof(double) * (size_t)imax);
    double* o = (double*)malloc(sizeof(double) * (size_t)H);
    orc_router_logits(x, T, H, router_w, E, logits);
    orc_route(logits, T, E, k, ids, w, probs);
    if (force_ids) {
        for (int t = 0; t < T; ++t) {
            double s = 0.0;
            for (int j = 0; j < k; ++j) {
                int e = force_ids[(size_t)t * k + j];
                ids[(size_t)t * k + j] = e;
                w[(size_t)t * k + j] = probs[(size_t)t * E + e];
                s += probs[(size_t)t * E + e];
            }
            for (int j = 0; j < k; ++j) w[(size_t)t * k + j] /= s;
        }
    }
    for (int t = 0; t < T && rc == ORC_OK; ++t) {
        double* yt = y + (size_t)t * H;
        for (int h = 0; h < H; ++h) { xv[h] = bf16_to_double(x[(size_t)t * H + h]); yt[h] = 0.0; }
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            if (!g_packed[e] || !u_packed[e] || !d_packed[e]) { rc = ORC_ERR_MISSING_EXPERT; break; }
            orc_mat g = {g_packed[e], g_scales[e], g_ts[e]};
            orc_mat u = {u_packed[e], u_scales[e], u_ts[e]};
            orc_mat d = {d_packed[e], d_scales[e], d_ts[e]};
            swiglu_expert(&g, &u, &d, kind, H, I, xv, ht, o);
            for (int h = 0; h < H; ++h) yt[h] += w[(size_t)t * k + j] * o[h];
        }
        if (rc != ORC_OK) break;
        double gate = 0.0;
        if (Is > 0) {
            for (int h = 0; h < H; ++h) gate += bf16_to_double(sh_gate_vec[h]) * xv[h];
            double sg = sigmoid(gate);
            orc_mat g = {sg_packed, sg_scales, sg_ts};
            orc_mat u = {su_packed, su_scales, su_ts};
            orc_mat d = {sd_packed, sd_scales, sd_ts};
            swiglu_expert(&g, &u, &d, kind, H, Is, xv, ht, o);
            for (int h = 0; h < H; ++h) yt[h] += sg * o[h];
            if (sig_out) sig_out[t] = sg;
        } else if (sig_out) {
            sig_out[t] = 0.0;
        }
    }
    if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)k * T);
    if (w_out) memcpy(w_out, w, sizeof(double) * (size_t)k * T);
    free(logits); free(probs); free(ids); free(w); free(xv); free(ht); free(o);
    return rc;
}

/* ------------------------------------------------------------ pre-MoE norm */

/* Round a double to the nearest bf16 (ties to even); returns the bf16 bits. Values
 * beyond bf16's range become +-inf, NaN stays NaN. Direct rounding from fp64 (no
 * intermediate fp32 step). */
uint16_t orc_bf16_from_double(double v) {
    if (isnan(v)) return 0x7FC0;
    int sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return (uint16_t)sign;
    /* bf16: 8 significant bits, exponent range of fp32 (normal min 2^-126, subnormal step 2^-133) */
    int ex;
    frexp(a, &ex);                       /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;                      /* a in [2^E, 2^(E+1)) */
    if (E < -126) E = -126;              /* subnormal: fixed quantum 2^-133 */
    double q = ldexp(a, 7 - E);          /* units of 2^(E-7) */
    double r = nearbyint(q);             /* ties to even (default rounding mode) */
    double back = ldexp(r, E - 7);
    if (back >= 0x1.FF8p127) return (uint16_t)(sign | 0x7F80);   /* rounds past the largest bf16 */
    /* encode back (exact in fp32) */
    float f = (float)back;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (u >> 16));
}

/* RMSNorm in the (1 + weight) form (lynn-engine tutorials index, row 01: RMSNorm =
 * (1.0 + weight) x x_norm; the Qwen 3.6 config block: rms_norm (1.0 + weight) x x_norm):
 *   x_norm[t,i] = h[t,i] / sqrt(mean_i h[t,i]^2 + eps),  out[t,i] = bf16((1 + w[i]) * x_norm[t,i])
 * All arithmetic in fp64; one rounding to bf16 (the activation type the layer consumes).
 * out_f64 (nullable) receives the value before that rounding. */
void orc_rmsnorm(const uint16_t* h, int T, int H, const uint16_t* w, double eps, uint16_t* out,
                 double* out_f64) {
    for (int t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int i = 0; i < H; ++i) {
            double v = bf16_to_double(h[(size_t)t * H + i]);
            ss += v * v;
        }
        double r = 1.0 / sqrt(ss / (double)H + eps);
        for (int i = 0; i < H; ++i) {
            double v = bf16_to_double(h[(size_t)t * H + i]) * r * (1.0 + bf16_to_double(w[i]));
            if (out_f64) out_f64[(size_t)t * H + i] = v;
            out[(size_t)t * H + i] = orc_bf16_from_double(v);
        }
    }
}
