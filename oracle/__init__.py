"""CPU oracle (test infrastructure only: tests, smoke() and bench.py's CPU leg)."""
from .oracle import *  # noqa: F401,F403
from .oracle import (decode_kdt, round_to_kdt, encode_kdt, ulp_kdt, num_pages, page_positions,
                     gather_rows, page_stats, cache_meta, head_meta, score_pages, select_pages,
                     select_pages_reserved, default_scale, attention, selected_positions,
                     merge_partials, page_decode_unit, h2o_fold, h2o_fold_window, h2o_store,
                     h2o_evict, h2o_unit_step, h2o_proxy_token, h2o_proxy_prefill, entmax_threshold, entmax,
                     attention_entmax, page_std, head_gauss_stats, gauss_page_moments,
                     gauss_global_moments, gauss_tail_moment, gauss_tau, gauss_max_factor,
                     gauss_select, gauss_decode_unit)
