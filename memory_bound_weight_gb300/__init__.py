"""GB300 (sm_103a) weight-streaming GEMV library: y = W.x and Y = X.W^T with
BF16, INT4 group-64 and AWQ-style INT4 group-128 weights."""
