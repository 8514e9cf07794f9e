"""The oracle: a plain, slow, FP64 CPU statement of the conditional-simulation hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import anything here.
The product path (the CUDA library and its Python binding) never imports, links or runs
this package, and this package never imports the product path.  The two share no code:
only the seeded input generators in ``inputgen`` serve both.

Every function follows "Mixed-Precision GPU Acceleration for Confidence Regions of
Spatial Excursion Sets" (Zhang, Abdulah, Cao, French, Alomairy, Genton, Keyes), cited by
section / equation / algorithm in each docstring.  Where the page is silent the plainest
reading is taken and named in the docstring.

Parity pins (tests/test_oracle_*.py) tie each function to something other than itself:
closed forms, library routines on special cases, brute force on tiny inputs and
invariants printed on the page.  Functions without such a pin say "parity unpinned".
"""
from .covariance import matern, powexp, covariance_fn, covariance_matrix, covariance_entries
from .policy import (PREC_FP64, PREC_FP32, PREC_FP16, tile_stats, tile_stats_from_locations,
                     precision_map, fp16_checks, covariance_scale, select_precision)
from .linalg import NotSPD, cholesky_lower, solve_lower, solve_lower_transpose
from .simulate import simulate, simulate_fp16_per_product, splitmix64, rnorm
from .krige import universal_kriging, conditional_correction
from .calibrate import (standardized_statistic, extrema_scan, exceedance_counts,
                        empirical_quantile, sample_without_sentinels, confidence_regions,
                        EmptySample, calibrate, calibrate_negative)
from .coverage import truth_field, excursion_set, coverage_event, inner_event, outer_event

__all__ = [
    "matern", "powexp", "covariance_fn", "covariance_matrix", "covariance_entries",
    "PREC_FP64", "PREC_FP32", "PREC_FP16", "tile_stats", "tile_stats_from_locations",
    "precision_map", "fp16_checks", "covariance_scale", "select_precision",
    "NotSPD", "cholesky_lower", "solve_lower", "solve_lower_transpose",
    "simulate", "simulate_fp16_per_product", "splitmix64", "rnorm", "universal_kriging", "conditional_correction",
    "standardized_statistic", "extrema_scan", "exceedance_counts", "empirical_quantile",
    "sample_without_sentinels", "confidence_regions", "EmptySample", "calibrate", "calibrate_negative",
    "truth_field", "excursion_set", "coverage_event", "inner_event", "outer_event",
]
