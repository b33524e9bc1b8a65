// The alpha / gamma planner: host arithmetic of "Fast Inference from
// Transformers via Speculative Decoding", section "方法细节" (期望生成 token
// 数, 墙钟加速因子, 运算量分析) and its FAQ on choosing gamma. No GPU work.

#include <cmath>

#include "specverify.h"

namespace {

bool alpha_ok(double a) { return a >= 0.0 && a <= 1.0; }

}  // namespace

extern "C" {

double spec_expected_tokens(double alpha, int gamma) {
    if (!alpha_ok(alpha) || gamma < 0) return NAN;
    if (alpha == 1.0) return gamma + 1.0;
    return (1.0 - std::pow(alpha, (double)(gamma + 1))) / (1.0 - alpha);
}

double spec_walltime_factor(double alpha, int gamma, double c) {
    if (!(c >= 0.0) || std::isinf(c)) return NAN;
    return spec_expected_tokens(alpha, gamma) / (gamma * c + 1.0);
}

double spec_ops_factor(double alpha, int gamma, double c_hat) {
    if (!(c_hat >= 0.0) || std::isinf(c_hat)) return NAN;
    return (gamma * c_hat + gamma + 1.0) / spec_expected_tokens(alpha, gamma);
}

int spec_best_gamma(double alpha, double c, int gamma_max) {
    if (!alpha_ok(alpha) || !(c >= 0.0) || std::isinf(c) || gamma_max < 1) return -1;
    double best = -1.0;
    int arg = 1;
    for (int g = 1; g <= gamma_max; ++g) {
        const double f = spec_walltime_factor(alpha, g, c);
        if (f > best) {
            best = f;
            arg = g;
        }
    }
    return arg;
}

}  // extern "C"
