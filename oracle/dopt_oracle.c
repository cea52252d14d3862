/*
 * Oracle for the ZeRO-1 distributed-optimizer step over a contiguous flat
 * gradient/parameter buffer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded CPU
 * statement of what the step computes.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg may build or call it.  It shares no
 * code, header or table with the CUDA library; the two are compared against
 * each other element by element.
 *
 * Sources (page titles and sections):
 *  [P1]  "04 · 分布式优化器" (Megatron-LM distributed optimizer)
 *        §2  the flat grad buffer cut into buckets; each bucket split into
 *            DP equal contiguous ranges, rank r owning range r.
 *        §3  the ownership demo: 1000 elements, DP 4, shard 250, rank 1 owns
 *            [250, 500); a param overlapping my range contributes the slice
 *            intersect(param range, my range).
 *        §4.1 Range(start, end) with normalize (rebase); the four ranges
 *            gbuf_world, gbuf_world_in_bucket, gbuf_local, param; every
 *            bucket size must divide by DP; rank r's range starts at
 *            r * (bucket size / DP).
 *        §4.2 reduce-scatter of each bucket: each rank keeps its 1/DP part.
 *        §4.3 the shard's grad goes to the fp32 main grad sliced by the
 *            "param" range; Adam runs on the shard only; the updated main
 *            shard is written back at gbuf_world_in_bucket.
 *        §4.4 all-gather of param_data gives every rank the full params.
 *        §5  gradient_scaling_factor multiplies the grads before the
 *            communication; padding keeps every bucket divisible by DP.
 *  [P2]  "distributed_training" tutorial, "AllReduce" (reduce-scatter then
 *        all-gather equals all-reduce), §8.2 mixed precision (bf16 model
 *        params, fp32 master weights) and §8.3 global norm clipping.
 *
 * Readings where the pages leave a step open (each one is listed in the
 * design notes of the repository):
 *  R1  Params sit at consecutive offsets in the order given; no per-param
 *      alignment.
 *  R2  Buckets are greedy: params are appended to the open bucket, which is
 *      closed as soon as its unpadded element count reaches bucket_elems
 *      (bucket_elems == 0: a single bucket).  A param never spans buckets.
 *      A bucket that holds at least one param is emitted.
 *  R3  Each bucket is padded at its end to a multiple of D * pad_unit; later
 *      buckets shift by that padding.  Padding belongs to no param and is
 *      never read or written by the step.
 *  R4  gbuf_world of a piece is the piece's own global range (all four
 *      ranges of a piece have the same length and differ by a translation).
 *  R5  Scaling: every replica element is widened to fp32 and multiplied by
 *      the fp32 scaling factor (one rounding) before the reduction; the
 *      reduction is fp32 in rank order, acc = x_0, acc = acc + x_r.
 *      The reduced fp32 value feeds Adam directly (no rounding to bf16).
 *  R6  Adam is AdamW with bias correction and decoupled decay, in fp32,
 *      each operation rounded once, in this order:
 *        m = b1*m + (1-b1)*g
 *        v = b2*v + (1-b2)*(g*g)
 *        w = w * (1 - lr*wd)                (only where the param decays)
 *        w = w - step_size * (m / (sqrt(v)/bc2_sqrt + eps))
 *      with step_size = lr/(1-b1^t) and bc2_sqrt = sqrt(1-b2^t).  The
 *      per-step scalars (1-b1), (1-b2), (1-lr*wd), step_size, bc2_sqrt are
 *      evaluated in double from the float hyper-parameters and rounded to
 *      float once.
 *  R7  Model params are bf16; fp32 -> bf16 is round-to-nearest-even, NaN
 *      stays a quiet NaN.
 *  R7b FP16 ([P2] §8.2 names FP16/BF16 for forward and backward; [P3]'s
 *      state table lists FP16 params and grads): grads may be IEEE binary16
 *      (widened exactly) and the model params binary16 too; fp32 -> fp16
 *      rounds to nearest even, overflows to Inf from 65520 on, and keeps
 *      subnormals.  Rounding the reduced grad (R12) and the all-reduce
 *      (R10) use the grads' type.
 *  R8  The all-gather copies every rank's owned elements (its pieces) from
 *      its own replica into all other replicas; padding is not copied.
 *  R9  Global-norm clipping ([P2] §8.3: the norm sqrt(sum ||g||^2) over all
 *      shards, needed before the optimizer update): norm^2 is the sum of the
 *      squares of the reduced fp32 grads of all owned elements, accumulated
 *      in double; the coefficient is min(1, max_norm / (norm + 1e-6)),
 *      evaluated in double and rounded to float once; each reduced grad is
 *      multiplied by it (one fp32 rounding) before Adam.
 *  R11 num_distributed_optimizer_instances ([P1] §5: the reduce-scatter
 *      stays inside an instance, an all-reduce across instances follows):
 *      the D ranks form `instances` groups of R = D / instances consecutive
 *      ranks; buckets are padded to and split into R ranges; each element's
 *      grad is, per instance, the rank-order fp32 sum of its R scaled
 *      replicas, and these sums are added in instance order.  Rank r of
 *      every instance computes the same update from the same state, so one
 *      copy of the optimizer state stands for all of them; the write-back
 *      goes to rank r of every instance and the all-gather runs inside each
 *      instance.
 *  R12 Optional (off by default): Megatron's reduce-scatter lands in the grad
 *      buffer ([P1] §4.2-§4.3: the shard is copied from the buffer to the
 *      main grads), so with that option the reduced grad is rounded to the
 *      grad type (bf16: R7) before clipping and Adam, and the norm is taken
 *      over the rounded grads.
 *  R13 Non-finite check (off by default).  [P2] §8.2 notes that FP16
 *      overflows easily; the pages give no rule for it, so the plain one is
 *      taken: an owned element is non-finite when its reduced grad (after
 *      the rounding of R12, when on) is Inf or NaN, counted once however
 *      many replicas contributed; padding is never counted; with the check
 *      on, a step with a non-zero count changes no state and no param (the
 *      caller simply does not step).  Scaling comes first (R5), so finite
 *      replicas whose unscaled sum would overflow are not counted when the
 *      scaled sum is finite.
 *  R10 force_all_reduce ([P1] §5) leaves the optimizer step unchanged (each
 *      rank still updates its own shard from the same reduced grads) and
 *      additionally gives every replica's grad buffer the whole reduced grad,
 *      rounded to the grad type.
 *
 * Windows: the step can be restricted to global buffer indices [w0, w1).
 * All buffer-indexed arrays passed to orc_step are then window-relative
 * (element i lives at index i - w0).  Elements are independent, so a window
 * gives exactly the values of the full computation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Grad element types (the grad_type arguments). */
#define ORC_GRAD_BF16 0
#define ORC_GRAD_F32 1
#define ORC_GRAD_F16 2

#define ORC_OK 0
#define ORC_E_ARG (-1)
#define ORC_E_LAYOUT (-2)
#define ORC_E_NOMEM (-6)

/* Range(start, end): half-open interval [start, end) ([P1] §4.1). */
typedef struct {
    int64_t start;
    int64_t end;
} orc_range;

/* One (param, rank) piece with its four ranges ([P1] §4.1 table). */
typedef struct {
    orc_range gbuf_world;
    orc_range gbuf_world_in_bucket;
    orc_range gbuf_local;
    orc_range param;
    int32_t param_id;
    int32_t bucket_id;
    int32_t rank;
    int32_t unused;
} orc_piece;

/* Range.normalize: the same interval translated to begin at `start`. */
static orc_range orc_normalize(orc_range r, int64_t start)
{
    orc_range out;
    out.start = start;
    out.end = start + (r.end - r.start);
    return out;
}

static int64_t orc_max(int64_t a, int64_t b) { return a > b ? a : b; }
static int64_t orc_min(int64_t a, int64_t b) { return a < b ? a : b; }

/* ------------------------------------------------------------------------ */
/* Layout: flat buffer, greedy buckets, padding (R1-R3).                    */
/* ------------------------------------------------------------------------ */

/*
 * param_start/param_end/param_bucket: [n].  bucket_start/bucket_end: room for
 * n buckets (a bucket holds at least one param).  Returns ORC_OK or an error.
 */
int orc_layout(const int64_t *sizes, int32_t n, int32_t D, int64_t bucket_elems,
               int32_t pad_unit, int64_t *param_start, int64_t *param_end,
               int32_t *param_bucket, int64_t *bucket_start, int64_t *bucket_end,
               int32_t *n_buckets_out, int64_t *numel_out)
{
    if (n < 0 || D < 1 || pad_unit < 1 || bucket_elems < 0)
        return ORC_E_ARG;
    for (int32_t p = 0; p < n; ++p)
        if (sizes[p] < 0)
            return ORC_E_ARG;

    int64_t unit = (int64_t)D * (int64_t)pad_unit;
    int64_t open_start = 0;  /* where the open bucket begins */
    int64_t open_count = 0;  /* unpadded elements in the open bucket */
    int32_t open_params = 0; /* params in the open bucket */
    int32_t nb = 0;

    for (int32_t p = 0; p < n; ++p) {
        param_start[p] = open_start + open_count;
        param_end[p] = param_start[p] + sizes[p];
        param_bucket[p] = nb;
        open_count += sizes[p];
        open_params += 1;
        if (bucket_elems > 0 && open_count >= bucket_elems) {
            int64_t padded = (open_count + unit - 1) / unit * unit;
            bucket_start[nb] = open_start;
            bucket_end[nb] = open_start + padded;
            nb += 1;
            open_start += padded;
            open_count = 0;
            open_params = 0;
        }
    }
    if (open_params > 0) {
        int64_t padded = (open_count + unit - 1) / unit * unit;
        bucket_start[nb] = open_start;
        bucket_end[nb] = open_start + padded;
        nb += 1;
        open_start += padded;
    }
    *n_buckets_out = nb;
    *numel_out = open_start;
    return ORC_OK;
}

/* Rank r's range in bucket k: [start + r*S, start + (r+1)*S), S = size/D
 * ([P1] §4.1, the per-rank ranges of each bucket). */
static int orc_rank_range(int64_t b_start, int64_t b_end, int32_t D, int32_t r,
                          orc_range *out)
{
    int64_t size = b_end - b_start;
    if (size % D != 0)
        return ORC_E_LAYOUT; /* the bucket-divides-by-DP assertion */
    int64_t S = size / D;
    out->start = b_start + (int64_t)r * S;
    out->end = out->start + S;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Four-way range map ([P1] §3 demo loop and §4.1).                         */
/* ------------------------------------------------------------------------ */

/*
 * For every bucket k, every rank r and every param p of bucket k (in order),
 * the overlap of p's buffer range with r's range gives one piece.  Pieces are
 * emitted sorted by (bucket, rank, gbuf_world.start).  `pieces` needs room
 * for n + D * n_buckets entries.
 */
int orc_pieces(int32_t n, const int64_t *param_start, const int64_t *param_end,
               const int32_t *param_bucket, int32_t nb, const int64_t *bucket_start,
               const int64_t *bucket_end, int32_t D, orc_piece *pieces,
               int32_t *n_pieces_out)
{
    int32_t np = 0;
    int32_t first = 0; /* the params of bucket k are consecutive from here */
    for (int32_t k = 0; k < nb; ++k) {
        while (first < n && param_bucket[first] < k)
            ++first;
        for (int32_t r = 0; r < D; ++r) {
            orc_range mine;
            int rc = orc_rank_range(bucket_start[k], bucket_end[k], D, r, &mine);
            if (rc != ORC_OK)
                return rc;
            for (int32_t p = first; p < n && param_bucket[p] == k; ++p) {
                int64_t x = orc_max(param_start[p], mine.start);
                int64_t y = orc_min(param_end[p], mine.end);
                if (x >= y)
                    continue;
                orc_piece pc;
                memset(&pc, 0, sizeof pc);
                pc.gbuf_world.start = x;
                pc.gbuf_world.end = y;
                pc.gbuf_world_in_bucket = orc_normalize(pc.gbuf_world, x - bucket_start[k]);
                pc.gbuf_local = orc_normalize(pc.gbuf_world, x - mine.start);
                pc.param = orc_normalize(pc.gbuf_world, x - param_start[p]);
                pc.param_id = p;
                pc.bucket_id = k;
                pc.rank = r;
                pieces[np++] = pc;
            }
        }
    }
    *n_pieces_out = np;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* bf16 helpers (R7).                                                       */
/* ------------------------------------------------------------------------ */

static float orc_bits_to_f32(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t orc_f32_to_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

float orc_bf16_to_f32(uint16_t h) { return orc_bits_to_f32((uint32_t)h << 16); }

/*
 * IEEE 754 binary16 (R7b): 1 sign bit, 5 exponent bits (bias 15), 10
 * fraction bits; exponent 0 holds zero and the subnormals (fraction *
 * 2^-24), exponent 31 Inf and NaN.  Widening to fp32 is exact.
 */
float orc_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t e = (h >> 10) & 0x1fu;
    uint32_t frac = h & 0x3ffu;
    if (e == 0x1fu)
        return orc_bits_to_f32(sign | 0x7f800000u | (frac << 13));
    if (e == 0) {
        float v = (float)frac * 0x1p-24f; /* exact: frac < 2^10 */
        return sign ? -v : v;
    }
    return orc_bits_to_f32(sign | ((e - 15u + 127u) << 23) | (frac << 13));
}

/*
 * fp32 -> binary16, round to nearest, ties to even; magnitudes from 65520
 * (the midpoint above the largest finite 65504, whose even neighbour is the
 * overflow) give Inf; NaN gives the quiet NaN 0x7e00 with the sign.  The
 * magnitude is divided by the quantum of its binade (a power of two, so
 * exactly, in double) and rounded with rint, which rounds ties to even in
 * the default rounding mode.
 */
uint16_t orc_f32_to_f16(float f)
{
    uint32_t u = orc_f32_to_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u)
        return (uint16_t)(sign | 0x7e00u);
    double ax = (double)orc_bits_to_f32(a);
    if (ax >= 65520.0)
        return (uint16_t)(sign | 0x7c00u);
    if (ax == 0.0)
        return sign;
    int e2 = 0;
    (void)frexp(ax, &e2); /* ax = m * 2^e2, 0.5 <= m < 1 */
    int ex = e2 - 1;      /* floor(log2 ax) */
    if (ex < -14)
        ex = -14;         /* the subnormals share the quantum 2^-24 */
    double n = rint(ldexp(ax, 10 - ex));
    if (n >= 2048.0) {
        n *= 0.5;
        ex += 1;
    }
    uint32_t bits;
    if (n >= 1024.0)
        bits = ((uint32_t)(ex + 15) << 10) | ((uint32_t)n - 1024u);
    else
        bits = (uint32_t)n; /* subnormal (ex == -14) */
    return (uint16_t)(sign | bits);
}

/* Round to nearest, ties to even, on the 16 dropped bits; NaN -> quiet NaN. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u = orc_f32_to_bits(f);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xffffu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u; /* may carry into the exponent: overflow gives inf */
    return (uint16_t)upper;
}

/* ------------------------------------------------------------------------ */
/* The step ([P1] §4.2-§4.4, readings R5-R8).                               */
/* ------------------------------------------------------------------------ */

typedef struct {
    float lr, beta1, beta2, eps, weight_decay, grad_scale;
} orc_adam;

/* Per-step scalars, each evaluated in double and rounded to float once (R6). */
typedef struct {
    float b1, b2, one_minus_b1, one_minus_b2, decay, step_size, bc2_sqrt, eps, scale;
} orc_scalars;

static orc_scalars orc_make_scalars(const orc_adam *c, int64_t t)
{
    orc_scalars s;
    double lr = c->lr, b1 = c->beta1, b2 = c->beta2, wd = c->weight_decay;
    s.b1 = c->beta1;
    s.b2 = c->beta2;
    s.one_minus_b1 = (float)(1.0 - b1);
    s.one_minus_b2 = (float)(1.0 - b2);
    s.decay = (float)(1.0 - lr * wd);
    s.step_size = (float)(lr / (1.0 - pow(b1, (double)t)));
    s.bc2_sqrt = (float)sqrt(1.0 - pow(b2, (double)t));
    s.eps = c->eps;
    s.scale = c->grad_scale;
    return s;
}

/* Element i of replica r, widened to fp32. */
static float orc_grad(const void *const *grads, int32_t grad_type, int32_t r, int64_t idx)
{
    if (grad_type == ORC_GRAD_F32)
        return ((const float *)grads[r])[idx];
    if (grad_type == ORC_GRAD_F16)
        return orc_f16_to_f32(((const uint16_t *)grads[r])[idx]);
    return orc_bf16_to_f32(((const uint16_t *)grads[r])[idx]);
}

/* The reduced grad of buffer element idx (R5, R11): inside each instance,
 * the rank-order fp32 sum of its R = D / instances scaled replicas (the
 * reduce-scatter within the instance); then the instances' sums added in
 * instance order (the all-reduce across instances).  With one instance this
 * is the plain rank-order sum.  `idx` is window-relative. */
static float orc_reduce_element(const void *const *grads, int32_t grad_type, int32_t D,
                                int32_t instances, float scale, int64_t idx)
{
    int32_t R = D / instances;
    float acc = 0.0f;
    for (int32_t inst = 0; inst < instances; ++inst) {
        int32_t first = inst * R;
        float part = scale * orc_grad(grads, grad_type, first, idx);
        for (int32_t q = first + 1; q < first + R; ++q) {
            float x = scale * orc_grad(grads, grad_type, q, idx);
            part = part + x;
        }
        acc = (inst == 0) ? part : acc + part;
    }
    return acc;
}

/* The reduced grad rounded to the grad buffer's type (R12): bf16 rounds to
 * nearest even (R7), fp32 stays as is. */
static float orc_round_to_grad_type(float g, int32_t grad_type)
{
    if (grad_type == ORC_GRAD_F16)
        return orc_f16_to_f32(orc_f32_to_f16(g));
    return grad_type == ORC_GRAD_F32 ? g : orc_bf16_to_f32(orc_f32_to_bf16(g));
}

/* One AdamW update of a single element (R6), fp32, one rounding per op. */
static void orc_adamw(const orc_scalars *s, int decays, float g, float *w, float *m, float *v)
{
    float mm = *m, vv = *v, ww = *w;
    float t1 = s->b1 * mm;
    float t2 = s->one_minus_b1 * g;
    mm = t1 + t2;
    float gg = g * g;
    float t3 = s->b2 * vv;
    float t4 = s->one_minus_b2 * gg;
    vv = t3 + t4;
    if (decays)
        ww = ww * s->decay;
    float root = sqrtf(vv);
    float corrected = root / s->bc2_sqrt;
    float denom = corrected + s->eps;
    float ratio = mm / denom;
    float delta = s->step_size * ratio;
    ww = ww - delta;
    *m = mm;
    *v = vv;
    *w = ww;
}

/*
 * One optimizer step for all D simulated ranks, restricted to the window
 * [w0, w1) of global buffer indices.
 *
 *   grads[D]        replica gradient buffers (bf16 bits or fp32), read only
 *   master, exp_avg, exp_avg_sq   fp32, buffer-indexed (element i of the
 *                   fp32 main params of the param that owns i)
 *   params[D]       replica bf16 param buffers (bits)
 *   gather          nonzero: all-gather into every replica (R8); zero: only
 *                   the owning rank's replica receives its updated shard
 *   main_grad_out   nullable: the reduce-scattered fp32 main grad of each
 *                   owned element, buffer-indexed (before clipping)
 *   clip_coef       global-norm clipping coefficient (orc_clip_coef); 1.0
 *                   when no clipping is wanted
 *   instances       optimizer instances (R11); D must divide by it; 1 is
 *                   the plain step
 *   round_grad      nonzero: the reduced grad is rounded to the grad type
 *                   before clipping and Adam (R12); main_grad_out then
 *                   reports the rounded value
 *
 * All buffer-indexed arrays are window-relative.  Returns ORC_OK or an error.
 */
int orc_step(const int64_t *sizes, int32_t n, const uint8_t *wd_mask, int32_t D,
             int32_t instances, int64_t bucket_elems, int32_t pad_unit,
             const orc_adam *cfg, int64_t step,
             int32_t grad_type, const void *const *grads, float *master, float *exp_avg,
             float *exp_avg_sq, uint16_t *const *params, int32_t gather,
             float *main_grad_out, int64_t w0, int64_t w1, float clip_coef,
             int32_t round_grad, int32_t param_is_f16)
{
    if (step < 1 || w0 < 0 || w1 < w0 || instances < 1 || D % instances != 0)
        return ORC_E_ARG;
    /* R ranks per instance shard each bucket (R11) */
    int32_t R = D / instances;

    int rc = ORC_OK;
    int64_t *pstart = NULL, *pend = NULL, *bstart = NULL, *bend = NULL;
    int32_t *pbucket = NULL;
    orc_piece *pieces = NULL;
    float *shard = NULL;
    int32_t nb = 0, npieces = 0;
    int64_t numel = 0;
    size_t cap = (size_t)(n > 0 ? n : 1);

    pstart = (int64_t *)malloc(cap * sizeof *pstart);
    pend = (int64_t *)malloc(cap * sizeof *pend);
    pbucket = (int32_t *)malloc(cap * sizeof *pbucket);
    bstart = (int64_t *)malloc(cap * sizeof *bstart);
    bend = (int64_t *)malloc(cap * sizeof *bend);
    if (!pstart || !pend || !pbucket || !bstart || !bend) {
        rc = ORC_E_NOMEM;
        goto done;
    }
    rc = orc_layout(sizes, n, R, bucket_elems, pad_unit, pstart, pend, pbucket, bstart,
                    bend, &nb, &numel);
    if (rc != ORC_OK)
        goto done;
    if (w1 > numel) {
        rc = ORC_E_ARG;
        goto done;
    }
    pieces = (orc_piece *)malloc(((size_t)n + (size_t)R * (size_t)nb + 1) * sizeof *pieces);
    if (!pieces) {
        rc = ORC_E_NOMEM;
        goto done;
    }
    rc = orc_pieces(n, pstart, pend, pbucket, nb, bstart, bend, R, pieces, &npieces);
    if (rc != ORC_OK)
        goto done;

    orc_scalars sc = orc_make_scalars(cfg, step);

    int32_t first_piece = 0;
    for (int32_t k = 0; k < nb; ++k) {
        for (int32_t r = 0; r < R; ++r) {
            orc_range mine = {0, 0};
            rc = orc_rank_range(bstart[k], bend[k], R, r, &mine);
            if (rc != ORC_OK)
                goto done;
            int64_t S = mine.end - mine.start;

            /* Reduce-scatter ([P1] §4.2, §5; R5, R11): rank r keeps the
             * scaled fp32 sum of its range over all D replicas. */
            free(shard);
            shard = (float *)malloc((size_t)(S > 0 ? S : 1) * sizeof *shard);
            if (!shard) {
                rc = ORC_E_NOMEM;
                goto done;
            }
            int64_t j_lo = orc_max(0, w0 - mine.start);
            int64_t j_hi = orc_min(S, w1 - mine.start);
            for (int64_t j = j_lo; j < j_hi; ++j) {
                int64_t i = mine.start + j;
                shard[j] = orc_reduce_element(grads, grad_type, D, instances, sc.scale,
                                              i - w0);
            }

            /* This rank's pieces are contiguous in the piece list. */
            int32_t last_piece = first_piece;
            while (last_piece < npieces && pieces[last_piece].bucket_id == k &&
                   pieces[last_piece].rank == r)
                ++last_piece;

            for (int32_t pi = first_piece; pi < last_piece; ++pi) {
                const orc_piece *pc = &pieces[pi];
                int32_t p = pc->param_id;
                int decays = wd_mask ? (wd_mask[p] != 0) : 1;
                int64_t t_lo = orc_max(0, w0 - pc->gbuf_world.start);
                int64_t t_hi = orc_min(pc->gbuf_world.end, w1) - pc->gbuf_world.start;
                for (int64_t t = t_lo; t < t_hi; ++t) {
                    int64_t i = pc->gbuf_world.start + t;
                    /* main grad: the shard sliced by gbuf_local ([P1] §4.3) */
                    float g = shard[pc->gbuf_local.start + t];
                    /* the reduced grad in the grad buffer's type (R12) */
                    if (round_grad)
                        g = orc_round_to_grad_type(g, grad_type);
                    /* global-norm clipping (R9): one fp32 multiply; a
                     * coefficient of exactly 1 leaves g unchanged */
                    float gc = g * clip_coef;
                    /* main param: the param's fp32 copy sliced by the "param"
                     * range; stored buffer-indexed at the param's offset. */
                    int64_t mi = pstart[p] + pc->param.start + t;
                    orc_adamw(&sc, decays, gc, &master[mi - w0], &exp_avg[mi - w0],
                              &exp_avg_sq[mi - w0]);
                    /* write-back into rank r's bucket view at
                     * gbuf_world_in_bucket ([P1] §4.3); rank r of every
                     * instance holds the same update (R11) */
                    int64_t bi = bstart[k] + pc->gbuf_world_in_bucket.start + t;
                    uint16_t updated = param_is_f16 ? orc_f32_to_f16(master[mi - w0])
                                                    : orc_f32_to_bf16(master[mi - w0]);
                    for (int32_t inst = 0; inst < instances; ++inst)
                        params[inst * R + r][bi - w0] = updated;
                    if (main_grad_out)
                        main_grad_out[i - w0] = g;
                }
            }

            /* All-gather ([P1] §4.4; R8): inside each instance, rank r's
             * owned elements go from its replica to the instance's other
             * replicas. */
            if (gather) {
                for (int32_t pi = first_piece; pi < last_piece; ++pi) {
                    const orc_piece *pc = &pieces[pi];
                    int64_t i_lo = orc_max(pc->gbuf_world.start, w0);
                    int64_t i_hi = orc_min(pc->gbuf_world.end, w1);
                    for (int64_t i = i_lo; i < i_hi; ++i) {
                        for (int32_t inst = 0; inst < instances; ++inst)
                            for (int32_t q = 0; q < R; ++q)
                                if (q != r)
                                    params[inst * R + q][i - w0] = params[inst * R + r][i - w0];
                    }
                }
            }
            first_piece = last_piece;
        }
    }

done:
    free(shard);
    free(pieces);
    free(pstart);
    free(pend);
    free(pbucket);
    free(bstart);
    free(bend);
    return rc;
}

/*
 * Number of owned elements of the window [w0, w1) whose reduced grad is Inf
 * or NaN (R13), after the optional rounding to the grad type (R12).  Grad
 * arrays are window-relative.
 */
int orc_count_nonfinite(const int64_t *sizes, int32_t n, int32_t D, int32_t instances,
                        int64_t bucket_elems, int32_t pad_unit, float grad_scale,
                        int32_t grad_type, const void *const *grads, int64_t w0, int64_t w1,
                        int32_t round_grad, int64_t *out)
{
    if (w0 < 0 || w1 < w0 || !out || instances < 1 || D % instances != 0)
        return ORC_E_ARG;
    int32_t R = D / instances;
    int rc = ORC_OK;
    size_t cap = (size_t)(n > 0 ? n : 1);
    int64_t *pstart = (int64_t *)malloc(cap * sizeof *pstart);
    int64_t *pend = (int64_t *)malloc(cap * sizeof *pend);
    int32_t *pbucket = (int32_t *)malloc(cap * sizeof *pbucket);
    int64_t *bstart = (int64_t *)malloc(cap * sizeof *bstart);
    int64_t *bend = (int64_t *)malloc(cap * sizeof *bend);
    orc_piece *pieces = NULL;
    int32_t nb = 0, npieces = 0;
    int64_t numel = 0;
    int64_t count = 0;
    if (!pstart || !pend || !pbucket || !bstart || !bend) {
        rc = ORC_E_NOMEM;
        goto done;
    }
    rc = orc_layout(sizes, n, R, bucket_elems, pad_unit, pstart, pend, pbucket, bstart, bend,
                    &nb, &numel);
    if (rc != ORC_OK)
        goto done;
    if (w1 > numel) {
        rc = ORC_E_ARG;
        goto done;
    }
    pieces = (orc_piece *)malloc(((size_t)n + (size_t)R * (size_t)nb + 1) * sizeof *pieces);
    if (!pieces) {
        rc = ORC_E_NOMEM;
        goto done;
    }
    rc = orc_pieces(n, pstart, pend, pbucket, nb, bstart, bend, R, pieces, &npieces);
    if (rc != ORC_OK)
        goto done;
    for (int32_t pi = 0; pi < npieces; ++pi) {
        int64_t i_lo = orc_max(pieces[pi].gbuf_world.start, w0);
        int64_t i_hi = orc_min(pieces[pi].gbuf_world.end, w1);
        for (int64_t i = i_lo; i < i_hi; ++i) {
            float r = orc_reduce_element(grads, grad_type, D, instances, grad_scale, i - w0);
            if (round_grad)
                r = orc_round_to_grad_type(r, grad_type);
            if (isinf(r) || isnan(r))
                ++count;
        }
    }
    *out = count;
done:
    free(pieces);
    free(pstart);
    free(pend);
    free(pbucket);
    free(bstart);
    free(bend);
    return rc;
}

/*
 * Sum of squares of the reduced grads over the owned elements of the window
 * [w0, w1) (R9), in piece order, accumulated in double.  Grad arrays are
 * window-relative.  Summing the results of disjoint windows that cover the
 * buffer gives the global norm^2.
 */
int orc_grad_norm_sq(const int64_t *sizes, int32_t n, int32_t D, int32_t instances,
                     int64_t bucket_elems, int32_t pad_unit, float grad_scale,
                     int32_t grad_type, const void *const *grads, int64_t w0, int64_t w1,
                     int32_t round_grad, double *out)
{
    if (w0 < 0 || w1 < w0 || !out || instances < 1 || D % instances != 0)
        return ORC_E_ARG;
    int32_t R = D / instances;
    int rc = ORC_OK;
    size_t cap = (size_t)(n > 0 ? n : 1);
    int64_t *pstart = (int64_t *)malloc(cap * sizeof *pstart);
    int64_t *pend = (int64_t *)malloc(cap * sizeof *pend);
    int32_t *pbucket = (int32_t *)malloc(cap * sizeof *pbucket);
    int64_t *bstart = (int64_t *)malloc(cap * sizeof *bstart);
    int64_t *bend = (int64_t *)malloc(cap * sizeof *bend);
    orc_piece *pieces = NULL;
    int32_t nb = 0, npieces = 0;
    int64_t numel = 0;
    double sum = 0.0;
    if (!pstart || !pend || !pbucket || !bstart || !bend) {
        rc = ORC_E_NOMEM;
        goto done;
    }
    rc = orc_layout(sizes, n, R, bucket_elems, pad_unit, pstart, pend, pbucket, bstart, bend,
                    &nb, &numel);
    if (rc != ORC_OK)
        goto done;
    if (w1 > numel) {
        rc = ORC_E_ARG;
        goto done;
    }
    pieces = (orc_piece *)malloc(((size_t)n + (size_t)R * (size_t)nb + 1) * sizeof *pieces);
    if (!pieces) {
        rc = ORC_E_NOMEM;
        goto done;
    }
    rc = orc_pieces(n, pstart, pend, pbucket, nb, bstart, bend, R, pieces, &npieces);
    if (rc != ORC_OK)
        goto done;
    for (int32_t pi = 0; pi < npieces; ++pi) {
        int64_t i_lo = orc_max(pieces[pi].gbuf_world.start, w0);
        int64_t i_hi = orc_min(pieces[pi].gbuf_world.end, w1);
        for (int64_t i = i_lo; i < i_hi; ++i) {
            float r = orc_reduce_element(grads, grad_type, D, instances, grad_scale, i - w0);
            if (round_grad)
                r = orc_round_to_grad_type(r, grad_type);
            double g = (double)r;
            sum += g * g;
        }
    }
    *out = sum;
done:
    free(pieces);
    free(pstart);
    free(pend);
    free(pbucket);
    free(bstart);
    free(bend);
    return rc;
}

/*
 * All-reduce of the grads ([P1] §5, force_all_reduce: every rank keeps the
 * whole reduced grad instead of its shard; [P2] "AllReduce": a
 * reduce-scatter followed by an all-gather).  For every (bucket, rank) the
 * shard is reduced as in the step (R5) and then written into every
 * replica's grad buffer at the shard's owned elements, rounded to the grad
 * type (R7 for bf16; fp32 stays as is) (R10).  Padding is not written.
 * grads are window-relative and are overwritten.
 */
int orc_allreduce(const int64_t *sizes, int32_t n, int32_t D, int32_t instances,
                  int64_t bucket_elems, int32_t pad_unit, float grad_scale, int32_t grad_type,
                  void *const *grads, int64_t w0, int64_t w1)
{
    if (w0 < 0 || w1 < w0 || instances < 1 || D % instances != 0)
        return ORC_E_ARG;
    int32_t R = D / instances;
    int rc = ORC_OK;
    size_t cap = (size_t)(n > 0 ? n : 1);
    int64_t *pstart = (int64_t *)malloc(cap * sizeof *pstart);
    int64_t *pend = (int64_t *)malloc(cap * sizeof *pend);
    int32_t *pbucket = (int32_t *)malloc(cap * sizeof *pbucket);
    int64_t *bstart = (int64_t *)malloc(cap * sizeof *bstart);
    int64_t *bend = (int64_t *)malloc(cap * sizeof *bend);
    orc_piece *pieces = NULL;
    float *shard = NULL;
    int32_t nb = 0, npieces = 0;
    int64_t numel = 0;
    if (!pstart || !pend || !pbucket || !bstart || !bend) {
        rc = ORC_E_NOMEM;
        goto done;
    }
    rc = orc_layout(sizes, n, R, bucket_elems, pad_unit, pstart, pend, pbucket, bstart, bend,
                    &nb, &numel);
    if (rc != ORC_OK)
        goto done;
    if (w1 > numel) {
        rc = ORC_E_ARG;
        goto done;
    }
    pieces = (orc_piece *)malloc(((size_t)n + (size_t)R * (size_t)nb + 1) * sizeof *pieces);
    if (!pieces) {
        rc = ORC_E_NOMEM;
        goto done;
    }
    rc = orc_pieces(n, pstart, pend, pbucket, nb, bstart, bend, R, pieces, &npieces);
    if (rc != ORC_OK)
        goto done;
    int32_t first_piece = 0;
    for (int32_t k = 0; k < nb; ++k) {
        for (int32_t r = 0; r < R; ++r) {
            orc_range mine = {0, 0};
            rc = orc_rank_range(bstart[k], bend[k], R, r, &mine);
            if (rc != ORC_OK)
                goto done;
            int64_t S = mine.end - mine.start;
            /* reduce-scatter: rank r's shard */
            free(shard);
            shard = (float *)malloc((size_t)(S > 0 ? S : 1) * sizeof *shard);
            if (!shard) {
                rc = ORC_E_NOMEM;
                goto done;
            }
            int64_t j_lo = orc_max(0, w0 - mine.start);
            int64_t j_hi = orc_min(S, w1 - mine.start);
            for (int64_t j = j_lo; j < j_hi; ++j)
                shard[j] = orc_reduce_element((const void *const *)grads, grad_type, D,
                                              instances, grad_scale, mine.start + j - w0);
            int32_t last_piece = first_piece;
            while (last_piece < npieces && pieces[last_piece].bucket_id == k &&
                   pieces[last_piece].rank == r)
                ++last_piece;
            /* all-gather of the shard into every replica's grad buffer */
            for (int32_t pi = first_piece; pi < last_piece; ++pi) {
                const orc_piece *pc = &pieces[pi];
                int64_t t_lo = orc_max(0, w0 - pc->gbuf_world.start);
                int64_t t_hi = orc_min(pc->gbuf_world.end, w1) - pc->gbuf_world.start;
                for (int64_t t = t_lo; t < t_hi; ++t) {
                    int64_t i = pc->gbuf_world.start + t;
                    float reduced = shard[pc->gbuf_local.start + t];
                    for (int32_t q = 0; q < D; ++q) {
                        if (grad_type == ORC_GRAD_F32)
                            ((float *)grads[q])[i - w0] = reduced;
                        else if (grad_type == ORC_GRAD_F16)
                            ((uint16_t *)grads[q])[i - w0] = orc_f32_to_f16(reduced);
                        else
                            ((uint16_t *)grads[q])[i - w0] = orc_f32_to_bf16(reduced);
                    }
                }
            }
            first_piece = last_piece;
        }
    }
done:
    free(shard);
    free(pieces);
    free(pstart);
    free(pend);
    free(pbucket);
    free(bstart);
    free(bend);
    return rc;
}

/* Clipping coefficient from the global norm^2 (R9). */
float orc_clip_coef(double norm_sq, float max_norm)
{
    double norm = sqrt(norm_sq);
    double coef = (double)max_norm / (norm + 1e-6);
    if (coef > 1.0)
        coef = 1.0;
    return (float)coef;
}

/* Convenience for tests: the layout and pieces in one call.  Sizes of the
 * outputs as in orc_layout / orc_pieces. */
int orc_range_map(const int64_t *sizes, int32_t n, int32_t D, int64_t bucket_elems,
                  int32_t pad_unit, int64_t *param_start, int64_t *param_end,
                  int32_t *param_bucket, int64_t *bucket_start, int64_t *bucket_end,
                  int32_t *n_buckets_out, int64_t *numel_out, orc_piece *pieces,
                  int32_t *n_pieces_out)
{
    int rc = orc_layout(sizes, n, D, bucket_elems, pad_unit, param_start, param_end,
                        param_bucket, bucket_start, bucket_end, n_buckets_out, numel_out);
    if (rc != ORC_OK)
        return rc;
    return orc_pieces(n, param_start, param_end, param_bucket, *n_buckets_out, bucket_start,
                      bucket_end, D, pieces, n_pieces_out);
}

/* The per-step scalars, for tests that pin them. */
void orc_step_scalars(const orc_adam *cfg, int64_t step, float *out9)
{
    orc_scalars s = orc_make_scalars(cfg, step);
    out9[0] = s.b1;
    out9[1] = s.b2;
    out9[2] = s.one_minus_b1;
    out9[3] = s.one_minus_b2;
    out9[4] = s.decay;
    out9[5] = s.step_size;
    out9[6] = s.bc2_sqrt;
    out9[7] = s.eps;
    out9[8] = s.scale;
}
