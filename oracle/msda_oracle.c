/*
 * msda_oracle.c -- TEST INFRASTRUCTURE, NOT THE PRODUCT.
 *
 * A plain, slow, obviously-correct CPU statement of multi-scale deformable
 * attention (MSDA), forward and backward, in IEEE binary64.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the CUDA
 * library never calls it and shares no code, header or table with it.
 *
 * What it follows:
 *   "MS Deformable Attention Kernel API Reference"
 *     - Background: every query/head samples each feature-pyramid level at
 *       learned normalised locations by bilinear interpolation and combines
 *       the samples with its attention weights.
 *     - Parameters: value (BLNC / BNLC), spatial_shapes (H_i, W_i),
 *       level_start_index, sampling_locations (BQHLP2 / B2QHLP),
 *       attention_weights (B, N_q, N_h, N_l, N_p), align_corners
 *       (True: [0,1] -> [0, H-1]; False: [0,1] -> [-0.5, H-0.5]),
 *       padding_mode ("zeros" / "border").
 *     - Returns: (B, N_q, N_h * C_h).
 *   "MS Deformable Attention Backward Kernel API Reference"
 *     - Background / Notes: gradients w.r.t. value, sampling_locations and
 *       attention_weights from bilinear-interpolation derivatives; "zeros":
 *       an out-of-bounds read is 0; "border": clamp to the edge.
 *     - Parameters: compute_grad_value / _sampling_locations /
 *       _attention_weights, at least one true.
 *     - Returns: grad_value (value's shape and layout), grad of
 *       sampling_locations (its shape and layout), grad_attention_weights
 *       (B, N_q, N_h, N_l, N_p).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - the trailing "2" of the location layouts is (x, y): x along W, y along H;
 *   - pixels of a level are flattened row-major: index = start + y*W + x;
 *   - output column = h*C_h + c;
 *   - "zeros" padding applies per bilinear corner (a corner outside the map
 *     reads 0), "border" clamps each corner's indices into the map;
 *   - the cell is chosen with floor(), so at an integer pixel coordinate the
 *     gradient is the one-sided derivative of the cell to the right.
 *
 * coord_f32: when non-zero, each pixel coordinate is rounded once to binary32
 * before the cell is chosen.  The sampling locations are binary32 inputs and
 * the GPU computes the pixel coordinate in binary32 with a single rounding;
 * this option lets the oracle take the same floor() decision so that
 * gradients (which jump across cell boundaries) are compared on the same cell.
 * With coord_f32 = 0 everything is exact binary64 (used by the pins).
 *
 * Parity status: every function here is pinned by the CPU tests (pixel-centre
 * identity, affine and bilinear closed forms, constant map, padding rules,
 * the one-level/one-point case against a library bilinear sampler, linearity,
 * layout permutations, grad_attention = <g, sample>, the adjoint identity,
 * and finite differences).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { LAYOUT_BLNC = 0, LAYOUT_BNLC = 1 };
enum { LAYOUT_BQHLP2 = 0, LAYOUT_B2QHLP = 1 };
enum { PAD_ZEROS = 0, PAD_BORDER = 1 };

typedef struct {
    int64_t B, N_q, N_h, C_h, N_l, N_p, L;
    const int64_t *shapes; /* N_l pairs (H_i, W_i) */
    const int64_t *starts; /* N_l entries */
    int value_layout, loc_layout, align_corners, padding_mode, coord_f32;
} problem;

/* Offset of value[b, pixel, h, c] ("value" parameter, both layouts). */
static int64_t value_offset(const problem *P, int64_t b, int64_t pix, int64_t h, int64_t c)
{
    if (P->value_layout == LAYOUT_BLNC)
        return ((b * P->L + pix) * P->N_h + h) * P->C_h + c;
    return ((b * P->N_h + h) * P->L + pix) * P->C_h + c;
}

/* Offset of coordinate xy (0 = x, 1 = y) of sample (b,q,h,l,p)
 * ("sampling_locations" parameter, both layouts). */
static int64_t loc_offset(const problem *P, int64_t b, int64_t q, int64_t h, int64_t l,
                          int64_t p, int xy)
{
    if (P->loc_layout == LAYOUT_BQHLP2)
        return (((((b * P->N_q + q) * P->N_h + h) * P->N_l + l) * P->N_p + p) * 2) + xy;
    return ((((b * 2 + xy) * P->N_q + q) * P->N_h + h) * P->N_l + l) * P->N_p + p;
}

/* Offset of attention_weights[b,q,h,l,p]. */
static int64_t attn_offset(const problem *P, int64_t b, int64_t q, int64_t h, int64_t l,
                           int64_t p)
{
    return (((b * P->N_q + q) * P->N_h + h) * P->N_l + l) * P->N_p + p;
}

/* Offset of out[b, q, h*C_h + c] (the returned (B, N_q, N_h*C_h) tensor). */
static int64_t out_offset(const problem *P, int64_t b, int64_t q, int64_t h, int64_t c)
{
    return (b * P->N_q + q) * (P->N_h * P->C_h) + h * P->C_h + c;
}

/* Normalised coordinate u in [0,1] -> pixel coordinate along an axis of
 * `size` pixels (align_corners parameter). */
static double pixel_coordinate(const problem *P, double u, int64_t size)
{
    double t = P->align_corners ? u * (double)(size - 1) : u * (double)size - 0.5;
    if (P->coord_f32)
        t = (double)(float)t;
    return t;
}

/* d(pixel coordinate)/du for the same mapping. */
static double pixel_scale(const problem *P, int64_t size)
{
    return P->align_corners ? (double)(size - 1) : (double)size;
}

/* The bilinear cell of one sample: four corners in the order
 * (y0,x0), (y0,x0+1), (y0+1,x0), (y0+1,x0+1), with their weights, the
 * derivatives of the weights w.r.t. the x and y pixel coordinates, whether
 * each corner reads the map, and the flattened pixel it reads. */
typedef struct {
    double w[4], dw_dx[4], dw_dy[4];
    int reads[4];
    int64_t pixel[4];
} cell;

static void make_cell(const problem *P, int64_t l, double x, double y, cell *k)
{
    const int64_t H = P->shapes[2 * l], W = P->shapes[2 * l + 1];
    const double x0 = floor(x), y0 = floor(y);
    const double fx = x - x0, fy = y - y0;
    const double cx[4] = {x0, x0 + 1.0, x0, x0 + 1.0};
    const double cy[4] = {y0, y0, y0 + 1.0, y0 + 1.0};
    const double wx[4] = {1.0 - fx, fx, 1.0 - fx, fx};
    const double wy[4] = {1.0 - fy, 1.0 - fy, fy, fy};
    const double dwx[4] = {-1.0, 1.0, -1.0, 1.0};
    const double dwy[4] = {-1.0, -1.0, 1.0, 1.0};
    for (int i = 0; i < 4; ++i) {
        k->w[i] = wx[i] * wy[i];
        k->dw_dx[i] = dwx[i] * wy[i];
        k->dw_dy[i] = wx[i] * dwy[i];
        double ix = cx[i], iy = cy[i];
        if (P->padding_mode == PAD_ZEROS) {
            k->reads[i] = (ix >= 0.0 && ix <= (double)(W - 1) && iy >= 0.0 && iy <= (double)(H - 1));
        } else {
            /* border: clamp the corner into the map */
            ix = ix < 0.0 ? 0.0 : (ix > (double)(W - 1) ? (double)(W - 1) : ix);
            iy = iy < 0.0 ? 0.0 : (iy > (double)(H - 1) ? (double)(H - 1) : iy);
            k->reads[i] = 1;
        }
        k->pixel[i] = k->reads[i] ? P->starts[l] + (int64_t)iy * W + (int64_t)ix : -1;
    }
}

static int check_problem(const problem *P)
{
    if (P->B < 0 || P->N_q < 0 || P->N_h < 0 || P->C_h < 0 || P->N_l < 0 || P->N_p < 0 || P->L < 0)
        return -1;
    int64_t s = 0;
    for (int64_t l = 0; l < P->N_l; ++l) {
        if (P->shapes[2 * l] < 1 || P->shapes[2 * l + 1] < 1 || P->starts[l] != s)
            return -1;
        s += P->shapes[2 * l] * P->shapes[2 * l + 1];
    }
    return s == P->L ? 0 : -1;
}

/* Forward: out[b,q,h*C_h+c] = sum_l sum_p A[b,q,h,l,p] * S_{b,q,h,l,p}[c],
 * S = sum over the four corners of w * value(corner). */
int msda_oracle_forward(int64_t B, int64_t N_q, int64_t N_h, int64_t C_h, int64_t N_l,
                        int64_t N_p, int64_t L, const int64_t *spatial_shapes,
                        const int64_t *level_start_index, int value_layout, int loc_layout,
                        int align_corners, int padding_mode, int coord_f32,
                        const double *value, const double *loc, const double *attn, double *out)
{
    const problem P = {B, N_q, N_h, C_h, N_l, N_p, L, spatial_shapes, level_start_index,
                       value_layout, loc_layout, align_corners, padding_mode, coord_f32};
    if (check_problem(&P))
        return -1;
    double *S = (double *)malloc(sizeof(double) * (size_t)(C_h > 0 ? C_h : 1));
    if (!S)
        return -2;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t q = 0; q < N_q; ++q)
            for (int64_t h = 0; h < N_h; ++h) {
                for (int64_t c = 0; c < C_h; ++c)
                    out[out_offset(&P, b, q, h, c)] = 0.0;
                for (int64_t l = 0; l < N_l; ++l) {
                    const int64_t H = spatial_shapes[2 * l], W = spatial_shapes[2 * l + 1];
                    for (int64_t p = 0; p < N_p; ++p) {
                        const double A = attn[attn_offset(&P, b, q, h, l, p)];
                        const double x = pixel_coordinate(&P, loc[loc_offset(&P, b, q, h, l, p, 0)], W);
                        const double y = pixel_coordinate(&P, loc[loc_offset(&P, b, q, h, l, p, 1)], H);
                        cell k;
                        make_cell(&P, l, x, y, &k);
                        for (int64_t c = 0; c < C_h; ++c)
                            S[c] = 0.0;
                        for (int i = 0; i < 4; ++i)
                            if (k.reads[i])
                                for (int64_t c = 0; c < C_h; ++c)
                                    S[c] += k.w[i] * value[value_offset(&P, b, k.pixel[i], h, c)];
                        for (int64_t c = 0; c < C_h; ++c)
                            out[out_offset(&P, b, q, h, c)] += A * S[c];
                    }
                }
            }
    free(S);
    return 0;
}

/* Backward, by the chain rule through the forward above.  With g the
 * grad_output row of (b,q,h) and v_i the value row read by corner i:
 *   grad_attention[s]   = <g, S_s>               = sum_i w_i <g, v_i>
 *   grad_loc_x[s]       = A_s * sum_i dw_i/dx <g, v_i> * dx/du
 *   grad_loc_y[s]       = A_s * sum_i dw_i/dy <g, v_i> * dy/du
 *   grad_value[corner] += A_s * w_i * g          (corners that read the map)
 * Disabled outputs are not touched.  grad_value is overwritten. */
int msda_oracle_backward(int64_t B, int64_t N_q, int64_t N_h, int64_t C_h, int64_t N_l,
                         int64_t N_p, int64_t L, const int64_t *spatial_shapes,
                         const int64_t *level_start_index, int value_layout, int loc_layout,
                         int align_corners, int padding_mode, int coord_f32,
                         const double *grad_output, const double *value, const double *loc,
                         const double *attn, int compute_grad_value,
                         int compute_grad_sampling_locations, int compute_grad_attention_weights,
                         double *grad_value, double *grad_loc, double *grad_attn)
{
    const problem P = {B, N_q, N_h, C_h, N_l, N_p, L, spatial_shapes, level_start_index,
                       value_layout, loc_layout, align_corners, padding_mode, coord_f32};
    if (check_problem(&P))
        return -1;
    if (!compute_grad_value && !compute_grad_sampling_locations && !compute_grad_attention_weights)
        return -3;
    if (compute_grad_value)
        for (int64_t i = 0; i < B * L * N_h * C_h; ++i)
            grad_value[i] = 0.0;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t q = 0; q < N_q; ++q)
            for (int64_t h = 0; h < N_h; ++h) {
                const double *g = grad_output + out_offset(&P, b, q, h, 0);
                for (int64_t l = 0; l < N_l; ++l) {
                    const int64_t H = spatial_shapes[2 * l], W = spatial_shapes[2 * l + 1];
                    for (int64_t p = 0; p < N_p; ++p) {
                        const double A = attn[attn_offset(&P, b, q, h, l, p)];
                        const double x = pixel_coordinate(&P, loc[loc_offset(&P, b, q, h, l, p, 0)], W);
                        const double y = pixel_coordinate(&P, loc[loc_offset(&P, b, q, h, l, p, 1)], H);
                        cell k;
                        make_cell(&P, l, x, y, &k);
                        /* <g, v_i> for each corner; 0 for a corner that reads nothing */
                        double gv[4] = {0.0, 0.0, 0.0, 0.0};
                        for (int i = 0; i < 4; ++i)
                            if (k.reads[i])
                                for (int64_t c = 0; c < C_h; ++c)
                                    gv[i] += g[c] * value[value_offset(&P, b, k.pixel[i], h, c)];
                        if (compute_grad_attention_weights) {
                            double s = 0.0;
                            for (int i = 0; i < 4; ++i)
                                s += k.w[i] * gv[i];
                            grad_attn[attn_offset(&P, b, q, h, l, p)] = s;
                        }
                        if (compute_grad_sampling_locations) {
                            double sx = 0.0, sy = 0.0;
                            for (int i = 0; i < 4; ++i) {
                                sx += k.dw_dx[i] * gv[i];
                                sy += k.dw_dy[i] * gv[i];
                            }
                            grad_loc[loc_offset(&P, b, q, h, l, p, 0)] = A * sx * pixel_scale(&P, W);
                            grad_loc[loc_offset(&P, b, q, h, l, p, 1)] = A * sy * pixel_scale(&P, H);
                        }
                        if (compute_grad_value)
                            for (int i = 0; i < 4; ++i)
                                if (k.reads[i])
                                    for (int64_t c = 0; c < C_h; ++c)
                                        grad_value[value_offset(&P, b, k.pixel[i], h, c)] +=
                                            A * k.w[i] * g[c];
                    }
                }
            }
    return 0;
}
