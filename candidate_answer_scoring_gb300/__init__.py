"""libjetscore: the candidate-set scoring head on one GB300 (sm_103a).

Hidden rows at teacher-forced candidate positions are projected onto the full
vocabulary inside a tcgen05/TMEM kernel that keeps a running log-sum-exp and
gathers only the supplied tokens' logits; candidate log-likelihoods, the set
softmax with temperature, the argmax decision, the expected index, confidence
and allowed-token mass follow in small kernels.  ``JetScorer`` is the Python
face of the C ABI in ``include/jetscore.h``.
"""
from .jetscore import (JET_ERR_ARG, JET_ERR_CUDA, JET_ERR_MODE, JET_ERR_NOT_IN_UNION,  # noqa: F401
                       JET_ERR_OFFSETS, JET_ERR_TIMEOUT, JET_ERR_TOKEN_RANGE, JET_ERR_UNSUPPORTED,
                       JET_ERR_WORKSPACE, JET_KIND_BINARY, JET_KIND_CHOICE, JET_KIND_ORDINAL, JET_MODE_FULL,
                       JET_MODE_RESTRICTED, JET_OK, JET_W_ROWMAJOR, JET_W_TILED, JetError, JetScorer, load,
                       status_string)
