"""GB300-native rollback-free tree verification for Gated DeltaNet layers.

Python face of libgdntree (C ABI in include/gdn_tree.h):

    o, U = verify(q, k, v, log_alpha, beta, parent, S0)
    S1   = commit(path, path_len, U, k, log_alpha, S0, parent=parent)
    S1, o, U = commit_verify(...)   # next iteration: commit fused into verify
    o, U = verify_recurrent(...)    # baseline: one recurrent pass per branch
    o, U = verify_packed(...)       # ragged batch, states in a pool (also commit_packed,
                                    # commit_verify_packed)
    parent, j, score, n = build_topw(cand_logp, w, max_depth)   # the draft tree

Build the library first with ``python -m gated_deltanet_tree_gdn_gb300.build``.
"""

from ._binding import (  # noqa: F401
    BF16, F32, OK, EINVAL, EUNSUPPORTED, ECUDA, STATUS_OK, STATUS_BAD_TREE,
    STATUS_BAD_PATH, STATUS_TIMEOUT, SYMBOLS, Dims, GdnTreeError, commit, commit_verify,
    library_path, load, strerror, verify, verify_recurrent, verify_packed, commit_packed,
    commit_verify_packed, STATUS_BAD_LAYOUT, build_topw,
)
from .build import build_library  # noqa: F401

__version__ = "0.1.0"
