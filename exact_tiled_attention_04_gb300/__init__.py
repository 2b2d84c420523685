"""GB300-native fused exact-attention forward pass (sm_103a).

O = softmax(scale * Q K^T) V and the per-row log-sum-exp, computed by one
fused CUDA kernel that never writes the N x N score matrix to HBM.
"""
